// Sage prepare for sm_103a: BF16 Q/K -> INT8 (per 32-row block scale), BF16 V ->
// FP8 e4m3 transposed (per channel scale), with optional QK RMSNorm and
// rotate-half RoPE first.  Follows the aiter pull request "gfx1201_sage_prepare
// / gfx1201_sage_attention" (commit message of gfx1201_sage_prepare; Technical
// Details).  Every binary32 operation uses an explicitly rounded intrinsic
// (no contraction), so the bytes written are a deterministic function of the
// inputs, and the order of the one order-dependent sum (RMSNorm's sum of
// squares) is fixed below.
//
// The per-element arithmetic (the RMSNorm factor and scaling, the RoPE pair, the
// codes and scales) is that of qk_quant.cuh, which the attention kernel's
// quantise-on-load of Q uses too, so both produce the same codes.  (NaN, which
// only RMSNorm of an all-zero or underflowing row with rms_eps = 0 produces, has
// no defined code.)
//
// Kernel 1 (tasks Q, K, V maxima over grid.z; Q or V may be skipped) -- one warp per (b, h, 32-row
// block).  A row of 128 channels is held by 8 lanes, lane L of the group owning
// channels [16L, 16L + 16) (two 128-bit loads); a warp covers 4 rows per step
// and 32 rows in 8 steps, so every lane keeps 8 rows x 16 channels in
// registers while the block maximum is reduced.  For V the same warps only
// take per-channel maxima, reduce them across the CTA and fold them into the
// workspace with integer atomicMax on the (non-negative) float bits.
// With K smoothing two kernels run first: per-block partial sums of K (same
// warp layout) and one thread per (b, h, channel) adding them up into the
// mean, which kernel 1 then subtracts from K.
// Kernel 2 -- one CTA per (b, h, 128 positions): 128 threads, thread (c8, sg)
// loads 16 positions x 8 channels, encodes them and transposes the bytes in
// registers (byte permutes) into 8 rows of 16 consecutive positions, which it
// writes with 128-bit stores into the [B, H, 128, S_pad] layout.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <mutex>
#include <type_traits>

#include "kernels.h"
#include "ptx.cuh"
#include "qk_quant.cuh"

namespace sa {
namespace {

struct QKParams {
  const __nv_bfloat16* x[3];
  long long sb[3], ss[3], sh[3];
  int B, S, H;
  long long S_pad;
  int nblk;                         // S_pad / 32
  const __nv_bfloat16* norm_w[2];   // Q, K (nullptr: no RMSNorm)
  float eps;
  const __nv_bfloat16* rope_cos;    // [S, rope_dim]
  const __nv_bfloat16* rope_sin;
  int rope_dim;
  int8_t* codes[2];
  __half* codes16[2];               // when set: the codes as FP16 (exact), [B*H, S_pad, 128], instead of INT8
  float* scales[2];
  float c_log2;                     // fl32(softmax_scale * log2 e), folded into Q's scales
  uint32_t* vmax;                   // [B*H*128] float bits of the channel maxima of |V|
  const float* kmean;               // [B*H*128] K smoothing: subtracted from K before quantising (or nullptr)
  __half* qmean16;                  // [B*H, S_pad/32, 128] Q smoothing: block means in step units (or nullptr)
  int task0;                        // task of grid.z = 0 (1 when Q is skipped)
};

using namespace qk;

__device__ __forceinline__ void unpack16(const uint32_t (&w)[8], float (&f)[16]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    f[2 * i] = bf_lo(w[i]);
    f[2 * i + 1] = bf_hi(w[i]);
  }
}
__device__ __forceinline__ void load16(const __nv_bfloat16* src, uint32_t (&w)[8]) {
  const uint4 a = __ldg(reinterpret_cast<const uint4*>(src));
  const uint4 b = __ldg(reinterpret_cast<const uint4*>(src) + 1);
  w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
  w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
}

// Rows row0 + 4*step + g (step < kSteps) of tensor `task` (0: Q, 1: K), channels
// [16L, 16L + 16), after the optional RMSNorm and RoPE, as packed BF16 pairs;
// rows >= S are zero.  A warp covers 4 * kSteps rows: a whole 32-row block
// (kSteps = 8) or half of one (4).  Shared by the quantiser and the K-mean
// partial sums, so both see the same bits.
template <int kSteps>
__device__ __forceinline__ void load_rows(const QKParams& p, int task, int bh, int row0, int lane,
                                          uint32_t (&x)[kSteps][8]) {
  const int b = bh / p.H, h = bh % p.H;
  const int g = lane >> 3;
  const int L = lane & 7;
  const __nv_bfloat16* base = p.x[task] + (long long)b * p.sb[task] + (long long)h * p.sh[task] + 16 * L;
  const long long ss = p.ss[task];
  // ---------------------------------------------------------- load kSteps rows x 16 channels
#pragma unroll
  for (int step = 0; step < kSteps; ++step) {
    const int s = row0 + 4 * step + g;
    if (s < p.S) {
      load16(base + (long long)s * ss, x[step]);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) x[step][i] = 0u;
    }
  }

  // ---------------------------------------------------------- RMSNorm (optional)
  const __nv_bfloat16* nw = p.norm_w[task];
  if (nw != nullptr) {
    uint32_t ww[8];
    load16(nw + 16 * L, ww);
    // the sum of squares of each row: 16-channel partials combined by an XOR butterfly (the
    // order of sumsq_combine, the same value in every lane of the row's group);
    // lane L of a group keeps the sum of its step-L row, takes 1 / sqrt(mean + eps) of it
    // once, and the group's lanes fetch each step's factor from lane L = step by a shuffle
    float mine = 0.0f;
#pragma unroll
    for (int step = 0; step < kSteps; ++step) {
      float acc = sumsq16(x[step]);
      acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, 4));
      acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, 2));
      acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, 1));
      mine = (L == step) ? acc : mine;
    }
    const float r_mine = rms_factor(mine, p.eps);
#pragma unroll
    for (int step = 0; step < kSteps; ++step) {
      const float r = __shfl_sync(0xffffffffu, r_mine, (lane & ~7) | step);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        x[step][i] = rms_apply(x[step][i], r, ww[i]);
    }
    // rows >= S stay exact zeros (with rms_eps = 0 their factor is infinite); only the last
    // block has such rows
    if (row0 + 4 * kSteps > p.S) {
#pragma unroll
      for (int step = 0; step < kSteps; ++step)
        if (row0 + 4 * step + g >= p.S)
#pragma unroll
          for (int i = 0; i < 8; ++i) x[step][i] = 0u;
    }
  }

  // ---------------------------------------------------------- rotate-half RoPE (optional)
  if (p.rope_dim > 0) {
    const int hh = p.rope_dim >> 1;
    const bool lo_half = 16 * L < hh;
    const bool in_rope = 16 * L < p.rope_dim;
    int src = lo_half ? L + (hh >> 4) : L - (hh >> 4);
    if (!in_rope) src = L;
    const int src_lane = (lane & ~7) | src;
    const uint32_t neg = lo_half ? 0x80008000u : 0u;
#pragma unroll
    for (int step = 0; step < kSteps; ++step) {
      uint32_t partner[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) partner[i] = __shfl_sync(0xffffffffu, x[step][i], src_lane);
      const int s = row0 + 4 * step + g;
      if (in_rope && s < p.S) {
        uint32_t cw[8], sw[8];
        load16(p.rope_cos + (long long)s * p.rope_dim + 16 * L, cw);
        load16(p.rope_sin + (long long)s * p.rope_dim + 16 * L, sw);
        // rope_first_half / rope_second_half, the half chosen per lane by the sign mask
#pragma unroll
        for (int i = 0; i < 8; ++i)
          x[step][i] = bf2_add(bf2_mul(x[step][i], cw[i]), bf2_mul(partner[i], sw[i]) ^ neg);
      }
    }
  }

}

// Grids of the per-block kernels: blockIdx.x = group of 8 blocks, blockIdx.y = head b * H + h
// (at most 65535 heads per launch: the launcher splits larger batches).
__device__ __forceinline__ void block_coords(int warp, int& bh, int& blk) {
  bh = (int)blockIdx.y;
  blk = (int)blockIdx.x * 8 + warp;
}

// The block's per-channel sums in the fixed order of the smoothing means: lane (g, L) adds
// its rows 32j + 4t + g over t = 0..7 (rows >= S hold +0, which changes nothing), then
//   B = (P_0 + P_1) + (P_2 + P_3)
// by two xor shuffles; every lane of channel group L ends with the block sums of its 16
// channels.
__device__ __forceinline__ void block_sums16(const uint32_t (&x)[8][8], float (&acc)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
#pragma unroll
  for (int step = 0; step < 8; ++step) {
    float f[16];
    unpack16(x[step], f);
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = __fadd_rn(acc[i], f[i]);
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    acc[i] = __fadd_rn(acc[i], __shfl_xor_sync(0xffffffffu, acc[i], 8));    // P_g + P_(g^1)
    acc[i] = __fadd_rn(acc[i], __shfl_xor_sync(0xffffffffu, acc[i], 16));   // + the other pair
  }
}

// Barrier 1 + group for the kWarps warps of one group (immediate ids, so that a kernel
// reserves only the barriers it names rather than all sixteen).
template <int kWarps>
__device__ __forceinline__ void group_bar_sync(int group) {
  switch (group) {
    case 0: asm volatile("bar.sync 1, %0;" ::"n"(32 * kWarps) : "memory"); break;
    case 1: asm volatile("bar.sync 2, %0;" ::"n"(32 * kWarps) : "memory"); break;
    case 2: asm volatile("bar.sync 3, %0;" ::"n"(32 * kWarps) : "memory"); break;
    default: asm volatile("bar.sync 4, %0;" ::"n"(32 * kWarps) : "memory"); break;
  }
}

// Blocks of 32 rows per CTA of the quantiser: the Q-smoothing instance gives each block
// one warp (its block sums run over all 32 rows of a lane group in a fixed order); the
// other gives each block two warps of 16 rows, which halves the rows a thread holds, so
// that four CTAs fit an SM instead of two: the kernel waits on HBM, and more resident
// warps keep more loads in flight (measured on a GB300: the prepare at Wan-720p 0.80 ->
// 0.71 ms, at FLUX-2048 with RMSNorm + RoPE 0.30 -> 0.26 ms; four warps of 8 rows at five
// CTAs per SM was slower at Wan-720p).
// Small problems (few blocks per task) take four warps of 8 rows per block instead, at
// five CTAs per SM: more and shorter CTAs fill the last wave of a small grid better
// (FLUX-1024, 3456 blocks per task: the one-call Sage op 195 -> 187 us; at 8192 blocks the
// prepare was already 5 % slower that way, and larger grids prefer two warps).
constexpr long long kQuantSmallBlocks = 4096;   // blocks per task (B * H * S_pad / 32) up to this
__host__ __device__ constexpr int quant_min_ctas(int warps_per_block) {
  return warps_per_block == 1 ? 1 : (warps_per_block == 2 ? 4 : 5);
}

// kWarpsPerBlock 1: the instance that smooths Q (its block mean, binary16 mean output)
template <int kWarpsPerBlock>
__global__ void __launch_bounds__(256, quant_min_ctas(kWarpsPerBlock)) prep_qk_vmax_kernel(const QKParams p) {
  griddep_launch_dependents();   // the next kernel may set up meanwhile (it waits for this grid)
  constexpr bool kQSmooth = (kWarpsPerBlock == 1);
  constexpr int kBlocksPerCta = 8 / kWarpsPerBlock;
  constexpr int kSteps = 8 / kWarpsPerBlock;          // rows per lane: 8, 4 or 2
  const int task = blockIdx.z + p.task0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = (int)blockIdx.y;
  const int blk = (int)blockIdx.x * kBlocksPerCta + warp / kWarpsPerBlock;
  const int half = warp % kWarpsPerBlock;             // which part of the block this warp holds
  const int row0 = 32 * blk + 4 * kSteps * half;      // this warp's first row
  const int b = bh / p.H, h = bh % p.H;
  const int g = lane >> 3;   // row inside a 4-row step
  const int L = lane & 7;    // channel group [16L, 16L+16)
  const __nv_bfloat16* base = p.x[task] + (long long)b * p.sb[task] + (long long)h * p.sh[task] + 16 * L;
  const long long ss = p.ss[task];

  if (task == 2) {
    // -------------------------------------------------------- V channel maxima
    __shared__ float red[8][128];
    uint32_t m2[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) m2[i] = 0u;
    if (blk < p.nblk) {
#pragma unroll
      for (int step = 0; step < kSteps; ++step) {
        const int s = row0 + 4 * step + g;
        if (s < p.S) {
          uint32_t w[8];
          load16(base + (long long)s * ss, w);
#pragma unroll
          for (int i = 0; i < 8; ++i) m2[i] = bf2_max(m2[i], bf2_abs(w[i]));
        }
      }
    }
    float mx[16];
    unpack16(m2, mx);
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      mx[k] = fmaxf(mx[k], __shfl_xor_sync(0xffffffffu, mx[k], 8));
      mx[k] = fmaxf(mx[k], __shfl_xor_sync(0xffffffffu, mx[k], 16));
    }
    if (g == 0) {
#pragma unroll
      for (int k = 0; k < 16; ++k) red[warp][16 * L + k] = mx[k];
    }
    __syncthreads();
    if (threadIdx.x < 128) {
      float m = red[0][threadIdx.x];
#pragma unroll
      for (int w2 = 1; w2 < 8; ++w2) m = fmaxf(m, red[w2][threadIdx.x]);
      if (m > 0.0f) atomicMax(&p.vmax[(long long)bh * 128 + threadIdx.x], __float_as_uint(m));
    }
    return;
  }

  if (blk >= p.nblk) return;   // (all warps of a block leave together)
  uint32_t x[kSteps][8];
  load_rows<kSteps>(p, task, bh, row0, lane, x);

  // ---------------------------------------------------------- K or Q smoothing (optional)
  // the value quantised is fl32(x - mean[channel]); it is formed again, bit for bit, for
  // the codes below.  K: the sequence mean from the smoothing kernels; Q: this block's own
  // mean, block sum / valid rows
  float mu[16];
  const bool qsmooth = kQSmooth && task == 0;
  const bool smooth = (task == 1 && p.kmean != nullptr) || qsmooth;
  bool have_mu = false;
  if constexpr (kQSmooth) {
    if (qsmooth) {
      block_sums16(x, mu);
      // valid rows; a block wholly past S has a zero sum and gets the mean +0
      const float n = (float)max(1, min(32, p.S - 32 * blk));
#pragma unroll
      for (int i = 0; i < 16; ++i) mu[i] = __fdiv_rn(mu[i], n);
      have_mu = true;
    }
  }
  if (!have_mu) {
#pragma unroll
    for (int i = 0; i < 16; ++i) mu[i] = smooth ? __ldg(p.kmean + (long long)bh * 128 + 16 * L + i) : 0.0f;
  }

  // ---------------------------------------------------------- block maximum and INT8 codes
  float a = 0.0f;
  if (smooth) {
#pragma unroll
    for (int step = 0; step < kSteps; ++step) {
      const int s = row0 + 4 * step + g;
      if (s < p.S) {
        float f[16];
        unpack16(x[step], f);
#pragma unroll
        for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(__fsub_rn(f[i], mu[i])));
      }
    }
  } else {
    // |x| of BF16 values is exact, so the maximum is taken on the BF16 pairs (rows >= S are 0)
    uint32_t m2 = 0u;
#pragma unroll
    for (int step = 0; step < kSteps; ++step)
#pragma unroll
      for (int i = 0; i < 8; ++i) m2 = bf2_max(m2, bf2_abs(x[step][i]));
    a = fmaxf(bf_lo(m2), bf_hi(m2));
  }
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, d));
  if constexpr (kWarpsPerBlock > 1) {
    // the block's maximum over its warps' parts: each posts its own, then a barrier of the
    // block's warps (named barrier 1 + block in the CTA; barrier 0 is left to __syncthreads)
    __shared__ float part_max[8];
    if (lane == 0) part_max[warp] = a;
    group_bar_sync<kWarpsPerBlock>(warp / kWarpsPerBlock);
    const int w0 = warp - half;
#pragma unroll
    for (int w2 = 0; w2 < kWarpsPerBlock; ++w2) a = fmaxf(a, part_max[w0 + w2]);
  }
  float inv;
  uint32_t m16[8];   // Q smoothing: the block mean in step units, binary16 pairs
  if (qsmooth) {
    // the step is at least max |mean| / (256 * 127), so that the mean in step units fits
    // binary16; a block whose 127 / a_eff overflows (below 127/FLT_MAX) is stored as zeros
    float cm = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) cm = fmaxf(cm, fabsf(mu[i]));
#pragma unroll
    for (int d = 4; d >= 1; d >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, d));
    a = fmaxf(a, __fmul_rn(cm, 1.0f / 256.0f));
    inv = code_factor(a);
    if (isinf(inv)) {
      inv = 0.0f;
      a = 0.0f;
#pragma unroll
      for (int i = 0; i < 16; ++i) mu[i] = 0.0f;   // stored as zeros: +0 means, not -0
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const __half2 h = __floats2half2_rn(__fmul_rn(mu[2 * i], inv), __fmul_rn(mu[2 * i + 1], inv));
      m16[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    if (g == 0) {
      uint4* dq = reinterpret_cast<uint4*>(p.qmean16 + ((long long)bh * p.nblk + blk) * 128 + 16 * L);
      dq[0] = make_uint4(m16[0], m16[1], m16[2], m16[3]);
      dq[1] = make_uint4(m16[4], m16[5], m16[6], m16[7]);
    }
  } else {
    inv = code_factor(a);
  }
  int8_t* out = p.codes[task] + ((long long)bh * p.S_pad) * 128 + 16 * L;
  __half* out16 = p.codes16[task] ? p.codes16[task] + ((long long)bh * p.S_pad) * 128 + 16 * L : nullptr;
  // codes by code_magic; its clamp only where 127 / a overflowed, a warp-uniform choice (the
  // block is one warp's)
  auto emit_codes = [&](auto kClamp, auto kSmooth) {
    constexpr bool kC = decltype(kClamp)::value;
#pragma unroll
    for (int step = 0; step < kSteps; ++step) {
      const int s = row0 + 4 * step + g;
      const bool live = s < p.S;
      auto code = [&](float f, int i) {
        if constexpr (decltype(kSmooth)::value) {
          return live ? code_magic<kC>(__fsub_rn(f, mu[i]), inv) : kRoundMagic;
        } else {
          return code_magic<kC>(f, inv);   // rows >= S hold zeros here, which code to 0
        }
      };
      if (out16) {
        // the same codes as FP16, exact: the operand the attention kernel's Q K^T MMA reads;
        // with Q smoothing, f16(code + mean) (one correctly rounded binary16 addition), which
        // carries the correction term mean . k into the same product
        uint32_t hw[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          hw[i] = codes_fp16x2(code(bf_lo(x[step][i]), 2 * i), code(bf_hi(x[step][i]), 2 * i + 1));
          if (qsmooth) {
            const __half2 sum = __hadd2(*reinterpret_cast<const __half2*>(&hw[i]),
                                        *reinterpret_cast<const __half2*>(&m16[i]));
            hw[i] = *reinterpret_cast<const uint32_t*>(&sum);
          }
        }
        uint4* d = reinterpret_cast<uint4*>(out16 + (long long)s * 128);
        d[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        d[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
      } else {
        uint32_t q[4];
#pragma unroll
        for (int w = 0; w < 4; ++w)
          q[w] = codes_int8x4(code(bf_lo(x[step][2 * w]), 4 * w), code(bf_hi(x[step][2 * w]), 4 * w + 1),
                              code(bf_lo(x[step][2 * w + 1]), 4 * w + 2), code(bf_hi(x[step][2 * w + 1]), 4 * w + 3));
        *reinterpret_cast<uint4*>(out + (long long)s * 128) = make_uint4(q[0], q[1], q[2], q[3]);
      }
    }
  };
  if (smooth) {
    if (isinf(inv)) emit_codes(std::true_type{}, std::true_type{});
    else emit_codes(std::false_type{}, std::true_type{});
  } else {
    if (isinf(inv)) emit_codes(std::true_type{}, std::false_type{});
    else emit_codes(std::false_type{}, std::false_type{});
  }
  if (lane == 0 && half == 0) p.scales[task][(long long)bh * p.nblk + blk] = block_scale(a, p.c_log2, task == 0);
}

// Q smoothing on the two-call path: Q's score operand f16(code + mean[block]) from the
// INT8 codes and the binary16 block means, 16 elements per thread and iteration (the
// rows of one head are consecutive, so global row / 32 is the block's index in qmean16).
__global__ void __launch_bounds__(256) widen_q_mean_kernel(const int8_t* __restrict__ q8,
                                                           const __half* __restrict__ qmean16,
                                                           __half* __restrict__ q16, long long n16) {
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152, 1152
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (long long)gridDim.x * blockDim.x) {
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(q8) + i);
    const long long e0 = 16 * i;                       // first element: row e0 / 128, channel e0 % 128
    const uint4* m4 = reinterpret_cast<const uint4*>(qmean16 + (e0 / 128 / 32) * 128 + (e0 % 128));
    const uint4 ma = __ldg(m4), mb = __ldg(m4 + 1);
    const uint32_t mw[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
    const uint32_t in[4] = {w.x ^ 0x80808080u, w.y ^ 0x80808080u, w.z ^ 0x80808080u, w.w ^ 0x80808080u};
    uint32_t out[8];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      // a byte u = code + 128 as the FP16 pattern 0x6400 | u is 1024 + u: minus 1152 is the code
      uint32_t lo = __byte_perm(in[t], 0x64646464u, 0x5140);
      uint32_t hi = __byte_perm(in[t], 0x64646464u, 0x7362);
      const __half2 hl = __hadd2(__hsub2(*reinterpret_cast<__half2*>(&lo), bias),
                                 *reinterpret_cast<const __half2*>(&mw[2 * t]));
      const __half2 hh = __hadd2(__hsub2(*reinterpret_cast<__half2*>(&hi), bias),
                                 *reinterpret_cast<const __half2*>(&mw[2 * t + 1]));
      out[2 * t] = *reinterpret_cast<const uint32_t*>(&hl);
      out[2 * t + 1] = *reinterpret_cast<const uint32_t*>(&hh);
    }
    uint4* d = reinterpret_cast<uint4*>(q16) + 2 * i;
    d[0] = make_uint4(out[0], out[1], out[2], out[3]);
    d[1] = make_uint4(out[4], out[5], out[6], out[7]);
  }
}

// ------------------------------------------------------------------ K smoothing
// mean[b, h, c] = (sum over s < S of K[b, s, h, c]) / S, K after the optional
// RMSNorm + RoPE, in a fixed binary32 order so that the mean (which decides
// INT8 codes) is a deterministic function of K.  Per 32-row block j the lanes
// g = 0..3 of a channel group hold rows 32j + 4t + g (t = 0..7):
//   P_g = (((0 + x[32j+g]) + x[32j+4+g]) + ...) + x[32j+28+g]
//   B_j = (P_0 + P_1) + (P_2 + P_3)                      (two xor shuffles)
// and the blocks are then added in ascending j from 0, and divided by S.
// Rows >= S load as +0, which leaves every sum unchanged.

// One warp per (b, h, block), as the quantiser: block sums B_j into partial[bh][j][128].
__global__ void __launch_bounds__(256) prep_kmean_partial_kernel(const QKParams p, float* __restrict__ partial) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int bh, blk;
  block_coords(warp, bh, blk);
  if (blk >= p.nblk) return;
  const int g = lane >> 3;
  const int L = lane & 7;
  uint32_t x[8][8];
  load_rows<8>(p, 1, bh, 32 * blk, lane, x);
  float acc[16];
  block_sums16(x, acc);
  if (g == 0) {
    float4* dst = reinterpret_cast<float4*>(partial + ((long long)bh * p.nblk + blk) * 128 + 16 * L);
#pragma unroll
    for (int v = 0; v < 4; ++v) dst[v] = make_float4(acc[4 * v], acc[4 * v + 1], acc[4 * v + 2], acc[4 * v + 3]);
  }
}

// One thread per (b, h, channel): the block sums in ascending order, then / S.
__global__ void __launch_bounds__(128) prep_kmean_kernel(const float* __restrict__ partial, int nblk, int S,
                                                         float* __restrict__ mean) {
  const int bh = blockIdx.x, c = threadIdx.x;
  const float* src = partial + (long long)bh * nblk * 128 + c;
  float total = 0.0f;
  for (int j = 0; j < nblk; ++j) total = __fadd_rn(total, __ldg(src + (long long)j * 128));
  mean[(long long)bh * 128 + c] = __fdiv_rn(total, (float)S);
}

struct VParams {
  const __nv_bfloat16* v;
  long long sb, ss, sh;
  int B, S, H;
  long long S_pad;
  const uint32_t* vmax;
  uint8_t* codes;   // [B, H, 128, S_pad]
  float* scales;    // [B, H, 128]
};

// 4 words (rows r..r+3, each holding 4 channel bytes, channel 0 lowest) ->
// 4 words (channels 0..3, each holding the 4 row bytes, row r lowest).
__device__ __forceinline__ void transpose4x4(uint32_t a, uint32_t b, uint32_t c, uint32_t d, uint32_t& o0,
                                             uint32_t& o1, uint32_t& o2, uint32_t& o3) {
  const uint32_t t0 = __byte_perm(a, b, 0x5140);  // a0 b0 a1 b1
  const uint32_t t1 = __byte_perm(a, b, 0x7362);  // a2 b2 a3 b3
  const uint32_t t2 = __byte_perm(c, d, 0x5140);  // c0 d0 c1 d1
  const uint32_t t3 = __byte_perm(c, d, 0x7362);  // c2 d2 c3 d3
  o0 = __byte_perm(t0, t2, 0x5410);               // a0 b0 c0 d0
  o1 = __byte_perm(t0, t2, 0x7632);               // a1 b1 c1 d1
  o2 = __byte_perm(t1, t3, 0x5410);
  o3 = __byte_perm(t1, t3, 0x7632);
}

// blockIdx.x = 128-position tile, blockIdx.y = head b * H + h
__global__ void __launch_bounds__(128) prep_v_kernel(const VParams p) {
  griddep_launch_dependents();
  griddep_wait();   // the channel maxima come from prep_qk_vmax_kernel
  const int bh = (int)blockIdx.y;
  const int tile = (int)blockIdx.x;
  const int b = bh / p.H, h = bh % p.H;
  const int c8 = threadIdx.x & 15;        // channels [8*c8, 8*c8 + 8)
  const int sg = threadIdx.x >> 4;        // positions [s0, s0 + 16)
  const long long s0 = (long long)tile * 128 + 16 * sg;

  float inv[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float a = __uint_as_float(p.vmax[(long long)bh * 128 + 8 * c8 + k]);
    inv[k] = (a > 0.0f) ? __fdiv_rn(448.0f, a) : 0.0f;
    if (tile == 0 && sg == 0) p.scales[(long long)bh * 128 + 8 * c8 + k] = (a > 0.0f) ? __fdiv_rn(a, 448.0f) : 0.0f;
  }

  const __nv_bfloat16* base = p.v + (long long)b * p.sb + (long long)h * p.sh + 8 * c8;
  uint32_t lo[16], hi[16];   // row r: channel bytes 0..3 and 4..7
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const long long s = s0 + r;
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (s < p.S) w = __ldg(reinterpret_cast<const uint4*>(base + s * p.ss));
    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
    float f[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __fmul_rn(bf_lo(wv[i]), inv[2 * i]);
      f[2 * i + 1] = __fmul_rn(bf_hi(wv[i]), inv[2 * i + 1]);
    }
    lo[r] = pack_e4m3x4(f[0], f[1], f[2], f[3]);
    hi[r] = pack_e4m3x4(f[4], f[5], f[6], f[7]);
  }
  uint32_t col[8][4];  // channel k, positions 4*t .. 4*t+3 in word t
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    transpose4x4(lo[4 * t], lo[4 * t + 1], lo[4 * t + 2], lo[4 * t + 3], col[0][t], col[1][t], col[2][t], col[3][t]);
    transpose4x4(hi[4 * t], hi[4 * t + 1], hi[4 * t + 2], hi[4 * t + 3], col[4][t], col[5][t], col[6][t], col[7][t]);
  }
  uint8_t* out = p.codes + ((long long)bh * 128 + 8 * c8) * p.S_pad + s0;
#pragma unroll
  for (int k = 0; k < 8; ++k)
    *reinterpret_cast<uint4*>(out + (long long)k * p.S_pad) = make_uint4(col[k][0], col[k][1], col[k][2], col[k][3]);
}

// Scratch of the allocation-free prepare entry point: the per-(b, h, channel)
// maxima of |V| for up to kNoAllocMaxHeads heads (B * H), 1 MiB in total.  It
// is a plain device global: every GPU that loads this library holds it until
// the process exits, and every call of that entry point on a device shares it.
__device__ __align__(256) static uint32_t g_prepare_scratch[kNoAllocMaxHeads * 128];

// e4m3 codes of n binary32 values (nearest even, saturating to +-448): four per
// thread through pack_e4m3x4, the packing of prep_v_kernel's V codes and of the
// attention kernel's FP8 P, so that the hardware conversion both rely on can be
// checked value by value.  Grid-stride; every access is guarded by n.
__global__ void __launch_bounds__(256) e4m3_encode_kernel(const float* __restrict__ x, uint8_t* __restrict__ y,
                                                          long long n) {
  const long long stride = 4LL * gridDim.x * blockDim.x;
  for (long long i = 4LL * ((long long)blockIdx.x * blockDim.x + threadIdx.x); i < n; i += stride) {
    float f[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) f[e] = i + e < n ? x[i + e] : 0.0f;
    const uint32_t w = pack_e4m3x4(f[0], f[1], f[2], f[3]);
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (i + e < n) y[i + e] = (uint8_t)(w >> (8 * e));
  }
}

}  // namespace

cudaError_t noalloc_prepare_scratch(uint32_t** out) {
  // In host code g_prepare_scratch only names the symbol.  Its device address belongs to
  // this library's module as loaded in one CUDA context, so it is looked up once per
  // context, with that context current, and cached under the context's id.
  static PerContext<uint32_t*> addr;
  return addr.get([](uint32_t** v) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_prepare_scratch);
    *v = static_cast<uint32_t*>(p);
    return e;
  }, out);
}

namespace {
// One launch sequence for at most 65535 heads (B * H).
cudaError_t launch_prepare_heads(const PrepareArgs& a, cudaStream_t stream) {
  const int nblk = (int)(a.S_pad / 32);
  cudaError_t e = cudaSuccess;
  if (!a.skip_v) {
    e = cudaMemsetAsync(a.vmax, 0, (size_t)a.B * a.H * 128 * sizeof(uint32_t), stream);
    if (e != cudaSuccess) return e;
  }
  QKParams p;
  for (int t = 0; t < 3; ++t) {
    p.x[t] = reinterpret_cast<const __nv_bfloat16*>(a.x[t]);
    p.sb[t] = a.str[t][0];
    p.ss[t] = a.str[t][1];
    p.sh[t] = a.str[t][2];
  }
  p.B = a.B;
  p.S = a.S;
  p.H = a.H;
  p.S_pad = a.S_pad;
  p.nblk = nblk;
  p.norm_w[0] = reinterpret_cast<const __nv_bfloat16*>(a.q_norm_w);
  p.norm_w[1] = reinterpret_cast<const __nv_bfloat16*>(a.k_norm_w);
  p.eps = a.rms_eps;
  p.rope_cos = reinterpret_cast<const __nv_bfloat16*>(a.rope_cos);
  p.rope_sin = reinterpret_cast<const __nv_bfloat16*>(a.rope_sin);
  p.rope_dim = a.rope_dim;
  p.codes[0] = a.q_i8;
  p.codes[1] = a.k_i8;
  p.codes16[0] = reinterpret_cast<__half*>(a.q16);
  p.codes16[1] = reinterpret_cast<__half*>(a.k16);
  p.scales[0] = a.q_scale;
  p.scales[1] = a.k_scale;
  p.c_log2 = a.c_log2;
  p.vmax = a.vmax;
  p.kmean = a.k_mean;
  p.qmean16 = reinterpret_cast<__half*>(a.q_mean16);
  p.task0 = a.skip_q ? (a.skip_k ? 2 : 1) : 0;
  // heads along grid.y (at most 65535 per launch, which the caller below guarantees)
  const int BH = a.B * a.H;
  if (a.k_mean != nullptr) {
    dim3 g0((nblk + 7) / 8, BH, 1);
    prep_kmean_partial_kernel<<<g0, 256, 0, stream>>>(p, a.k_partial);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    prep_kmean_kernel<<<BH, 128, 0, stream>>>(a.k_partial, nblk, a.S, a.k_mean);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // tasks [task0, 3 or 2) over grid.z (none left when the forward codes Q and K and V is
  // not quantised)
  const int tasks = (a.skip_v ? 2 : 3) - p.task0;
  if (tasks > 0) {
    const bool q_smooth = p.qmean16 != nullptr && p.task0 == 0;
    const int wpb = q_smooth ? 1 : ((long long)BH * nblk <= kQuantSmallBlocks ? 4 : 2);
    const int per_cta = 8 / wpb;
    dim3 g1((nblk + per_cta - 1) / per_cta, BH, tasks);
    if (wpb == 1)
      prep_qk_vmax_kernel<1><<<g1, 256, 0, stream>>>(p);
    else if (wpb == 2)
      prep_qk_vmax_kernel<2><<<g1, 256, 0, stream>>>(p);
    else
      prep_qk_vmax_kernel<4><<<g1, 256, 0, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (a.skip_v) return cudaSuccess;

  VParams vp;
  vp.v = reinterpret_cast<const __nv_bfloat16*>(a.x[2]);
  vp.sb = a.str[2][0];
  vp.ss = a.str[2][1];
  vp.sh = a.str[2][2];
  vp.B = a.B;
  vp.S = a.S;
  vp.H = a.H;
  vp.S_pad = a.S_pad;
  vp.vmax = a.vmax;
  vp.codes = a.v_fp8;
  vp.scales = a.v_scale;
  dim3 g2((unsigned)(a.S_pad / 128), BH, 1);
  // a programmatic dependent of prep_qk_vmax_kernel (it waits before reading the maxima)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = g2;
  cfg.blockDim = dim3(128, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prep_v_kernel, vp);
}

}  // namespace

cudaError_t launch_sage_prepare(const PrepareArgs& a, cudaStream_t stream) {
  constexpr long long kMaxHeads = 65535;   // grid.y of the prepare kernels
  if ((long long)a.B * a.H <= kMaxHeads) return launch_prepare_heads(a, stream);
  if (a.H > kMaxHeads) return cudaErrorInvalidConfiguration;
  // more heads than one grid holds: whole batch entries at a time, every pointer moved to
  // the chunk's first batch entry (all per-head outputs are indexed by b * H + h)
  const int per = (int)(kMaxHeads / a.H);
  const long long S_pad = a.S_pad, nblk = S_pad / 32;
  for (int b0 = 0; b0 < a.B; b0 += per) {
    PrepareArgs c = a;
    c.B = a.B - b0 < per ? a.B - b0 : per;
    const long long h0 = (long long)b0 * a.H;   // first head of the chunk
    for (int t = 0; t < 3; ++t)
      c.x[t] = static_cast<const __nv_bfloat16*>(a.x[t]) + (long long)b0 * a.str[t][0];
    auto bytes = [](void* p, long long off) { return p ? static_cast<void*>(static_cast<uint8_t*>(p) + off) : p; };
    c.q_i8 = static_cast<int8_t*>(bytes(a.q_i8, h0 * S_pad * 128));
    c.k_i8 = static_cast<int8_t*>(bytes(a.k_i8, h0 * S_pad * 128));
    c.v_fp8 = static_cast<uint8_t*>(bytes(a.v_fp8, h0 * 128 * S_pad));
    c.q16 = bytes(a.q16, h0 * S_pad * 128 * 2);
    c.k16 = bytes(a.k16, h0 * S_pad * 128 * 2);
    c.q_scale = static_cast<float*>(bytes(a.q_scale, h0 * nblk * 4));
    c.k_scale = static_cast<float*>(bytes(a.k_scale, h0 * nblk * 4));
    c.v_scale = static_cast<float*>(bytes(a.v_scale, h0 * 128 * 4));
    c.vmax = static_cast<uint32_t*>(bytes(a.vmax, h0 * 128 * 4));
    c.k_mean = static_cast<float*>(bytes(a.k_mean, h0 * 128 * 4));
    c.k_partial = static_cast<float*>(bytes(a.k_partial, h0 * nblk * 128 * 4));
    c.q_mean16 = bytes(a.q_mean16, h0 * nblk * 128 * 2);
    cudaError_t e = launch_prepare_heads(c, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_widen_q_mean(const int8_t* q8, const void* qmean16, void* q16, long long n_codes, int num_sms,
                               cudaStream_t stream) {
  const long long n16 = n_codes / 16;
  long long blocks = (n16 + 255) / 256;
  const long long cap = (long long)num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  widen_q_mean_kernel<<<(unsigned)blocks, 256, 0, stream>>>(q8, reinterpret_cast<const __half*>(qmean16),
                                                             reinterpret_cast<__half*>(q16), n16);
  return cudaGetLastError();
}

cudaError_t launch_e4m3_encode(const float* x, uint8_t* y, long long n, int num_sms, cudaStream_t stream) {
  long long blocks = (n + 4LL * 256 - 1) / (4LL * 256);
  const long long cap = (long long)num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  e4m3_encode_kernel<<<(unsigned)blocks, 256, 0, stream>>>(x, y, n);
  return cudaGetLastError();
}

}  // namespace sa
