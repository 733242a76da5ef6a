// Non-causal flash attention forward, BF16 in / BF16 out, head dim 128, for sm_103a.
//
// What it computes: O = softmax(scale * Q K^T) V per (batch, head), streaming
// K/V tiles and keeping a running row maximum, a running row sum and an
// unnormalised FP32 accumulator, rescaled when the maximum grows, divided by
// the sum at the end -- the tiled online softmax of the ai-infra handbook
// chapter "Kernel acceleration: attention, compilation and fusion" (section
// "Attention: from O(N^2) memory to blocks", the blocked form) and of the
// RDNA2 DiT flash kernel note (Contribution: "tiled, online-softmax, no full
// attention matrix materialized").  Exponentials are taken base 2 with
// scale*log2(e) folded into the scores, which is the same function.
//
// How (one CTA = one (batch, head) and two 128-row Q tiles, 320 threads):
//   warp 8      TMA producer: Q tiles once, then K_j, V_j into a 4-slot ring
//   warp 9      MMA issuer:   S_i = Q_i K_j^T and O_i += P_i V_j on tcgen05
//                             (kind::f16, FP32 accumulators in TMEM)
//   warps 0-7   softmax: warps 0-3 own key columns [0,64) and warps 4-7 key
//               columns [64,128) of every score tile (one thread per row and
//               half-row, TMEM lane = row); both warpgroups take Q tile 0 then
//               Q tile 1 each step and exchange half-row maxima in shared memory
// TMEM columns: S_0 [0,128), S_1 [128,256), O_0 [256,384), O_1 [384,512);
// P_i (BF16, two per column) overwrites the first 64 columns of S_i and is
// the A operand of the PV MMA straight from TMEM, each warpgroup writing the
// half of P for its key columns.  The two Q tiles ping-pong: while the softmax
// warps exponentiate S_0, the tensor core runs S_1 and P V.  Splitting each
// tile's columns over both warpgroups halves the time from a tile's scores to
// its P, which is the chain that bounds the kernel (scores done -> softmax ->
// P V -> next scores of that tile).
// Rescaling is lazy: the reference maximum of a row moves only when a tile's
// maximum exceeds it by more than kTau (log2 units), so P <= 2^kTau and O
// is rescaled rarely; the final division uses the same reference, so the
// result is unchanged.
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"

namespace sa {
namespace {

constexpr int kBM = 128;               // rows per Q tile
constexpr int kBN = 128;               // keys per K/V tile
constexpr int kNQ = 2;                 // Q tiles per CTA
constexpr int kStages = 4;             // K/V ring slots
constexpr int kTileBytes = 128 * 128 * 2;   // one BF16 128x128 tile
constexpr int kHalfBytes = kTileBytes / 2;  // [128 rows][64 columns] sub-tile, one 128B-swizzled TMA box
constexpr int kThreads = 320;
constexpr int kWarpLoad = 8;
constexpr int kWarpMma = 9;
constexpr float kTau = 8.0f;

struct __align__(1024) Smem {
  uint8_t q[kNQ][kTileBytes];
  uint8_t kv[kStages][kTileBytes];
  uint64_t q_full;
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full[kNQ];
  uint64_t p_full[kNQ][2];   // P_i keys [0,64) and [64,128) stored in TMEM
  uint64_t o_done[kNQ];
  uint64_t xch[kNQ];         // half-row maxima of Q tile i exchanged (all 8 softmax warps)
  uint64_t xfin[kNQ];        // half-row sums of Q tile i exchanged (epilogue)
  float xmax[kNQ][2][kBM];   // half-row maxima, [tile][column half][row]
  float xsum[kNQ][2][kBM];   // half-row sums
  uint64_t mma_drain;
  uint32_t tmem_base;
  uint32_t abort_flag;
};

__device__ uint32_t g_err_bf16;

struct Params {
  __nv_bfloat16* o;
  long long o_sb, o_ss, o_sh;
  int S;
  int n_tiles;
  float c_log2;  // softmax_scale * log2(e)
};

__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }
__device__ __forceinline__ uint32_t f2u(float f) { return __float_as_uint(f); }

__global__ void __launch_bounds__(kThreads, 1)
    attn_bf16_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.y, b = blockIdx.z;
  const int q_row0 = blockIdx.x * (kNQ * kBM);
  const int n = p.n_tiles;
  volatile uint32_t* abort_flag = &sm.abort_flag;

  if (threadIdx.x == 0) {
    mbar_init(&sm.q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.kv_full[s], 1);
      mbar_init(&sm.kv_empty[s], 1);
    }
    for (int i = 0; i < kNQ; ++i) {
      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.p_full[i][0], 4);
      mbar_init(&sm.p_full[i][1], 4);
      mbar_init(&sm.o_done[i], 1);
      mbar_init(&sm.xch[i], 8);
      mbar_init(&sm.xfin[i], 8);
    }
    mbar_init(&sm.mma_drain, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == kWarpLoad) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(&sm.q_full, kNQ * kTileBytes);
      for (int i = 0; i < kNQ; ++i)
        for (int hf = 0; hf < 2; ++hf)
          tma_load_4d(sm.q[i] + hf * kHalfBytes, &tm_q, &sm.q_full, hf * 64, q_row0 + i * kBM, h, b);
      int issued = 0;
      bool ok = true;
      for (int j = 0; j < n && ok; ++j) {
        for (int t = 0; t < 2; ++t) {
          const int item = 2 * j + t, slot = item % kStages, use = item / kStages;
          if (use > 0 && !mbar_wait(&sm.kv_empty[slot], (use - 1) & 1, abort_flag, &g_err_bf16, kErrTimeoutSync)) {
            ok = false;
            break;
          }
          const CUtensorMap* tm = (t == 0) ? &tm_k : &tm_v;
          mbar_arrive_expect_tx(&sm.kv_full[slot], kTileBytes);
          tma_load_4d(sm.kv[slot], tm, &sm.kv_full[slot], 0, j * kBN, h, b);
          tma_load_4d(sm.kv[slot] + kHalfBytes, tm, &sm.kv_full[slot], 64, j * kBN, h, b);
          issued = item + 1;
        }
      }
      if (*abort_flag) {
        // let copies in flight land before the CTA's shared memory goes away
        mbar_wait_teardown(&sm.q_full, 0);
        for (int item = (issued > kStages ? issued - kStages : 0); item < issued; ++item)
          mbar_wait_teardown(&sm.kv_full[item % kStages], (item / kStages) & 1);
      }
    }
  } else if (warp == kWarpMma) {
    {
      // the whole warp runs the issue loop (descriptors and loop state stay
      // warp-uniform, which keeps each tcgen05.mma issue cheap); one elected
      // lane issues every tcgen05 instruction
      const bool leader = elect_one();
      // ------------------------------------------------------------ MMA issuer
      const uint32_t idesc_qk = idesc_f32acc(kFmtBF16, kFmtBF16, false, false, kBM, kBN);
      const uint32_t idesc_pv = idesc_f32acc(kFmtBF16, kFmtBF16, false, true, kBM, 128);
      // TMEM columns of S_i and O_i
      auto tS = [&](int i) { return tmem + 128u * (uint32_t)i; };
      auto tO = [&](int i) { return tmem + 256u + 128u * (uint32_t)i; };
      uint32_t* err = &g_err_bf16;

      auto issue_s = [&](int i, int slot) {
        const uint32_t qa = smem_u32(sm.q[i]), ka = smem_u32(sm.kv[slot]);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
          const uint64_t da = smem_desc_sw128(qa + off, 16, 1024), db = smem_desc_sw128(ka + off, 16, 1024);
          if (leader) mma_f16_ss(tS(i), da, db, idesc_qk, kk > 0 ? 1u : 0u);
        }
      };
      // O_i += P_i V for keys [64*half, 64*half + 64): 4 steps of 16 keys, i.e. rows
      // kk*16.. of the [key][d] tile; the two 64-column halves of d sit kHalfBytes
      // apart (LBO), 8-row groups 1024 bytes apart (SBO)
      auto issue_pv_half = [&](int i, int slot, int half, bool acc) {
        const uint32_t va = smem_u32(sm.kv[slot]);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const int kk = 4 * half + k4;
          const uint64_t db = smem_desc_sw128(va + kk * 2048, kHalfBytes, 1024);
          if (leader) mma_f16_ts(tO(i), tS(i) + kk * 8, db, idesc_pv, (acc || kk > 0) ? 1u : 0u);
        }
      };
      // wait for each half of P_i, issue its four MMAs, then signal O_i done
      auto issue_pv = [&](int i, int slot, int j) -> bool {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          if (!mbar_wait_warp(&sm.p_full[i][half], j & 1, abort_flag, err, kErrTimeoutSync)) return false;
          tc_fence_after();
          issue_pv_half(i, slot, half, j > 0);
        }
        if (leader) mma_commit(&sm.o_done[i]);
        return true;
      };

      bool ok = mbar_wait_warp(&sm.q_full, 0, abort_flag, err, kErrTimeoutTma);
      if (ok) ok = mbar_wait_warp(&sm.kv_full[0], 0, abort_flag, err, kErrTimeoutTma);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        if (leader) mma_commit(&sm.s_full[0]);
        issue_s(1, 0);
        if (leader) mma_commit(&sm.s_full[1]);
        if (leader) mma_commit(&sm.kv_empty[0]);
      }
      for (int j = 0; j < n && ok; ++j) {
        const int itV = 2 * j + 1, slotV = itV % kStages;
        const int itK = 2 * j + 2, slotK = itK % kStages;
        const bool more = (j + 1 < n);
        if (!mbar_wait_warp(&sm.kv_full[slotV], (itV / kStages) & 1, abort_flag, err, kErrTimeoutTma)) break;
        if (!issue_pv(0, slotV, j)) break;
        if (more) {
          if (!mbar_wait_warp(&sm.kv_full[slotK], (itK / kStages) & 1, abort_flag, err, kErrTimeoutTma)) break;
          tc_fence_after();
          issue_s(0, slotK);
          if (leader) mma_commit(&sm.s_full[0]);
        }
        if (!issue_pv(1, slotV, j)) break;
        if (leader) mma_commit(&sm.kv_empty[slotV]);
        if (more) {
          issue_s(1, slotK);
          if (leader) mma_commit(&sm.s_full[1]);
          if (leader) mma_commit(&sm.kv_empty[slotK]);
        }
      }
      // every MMA the leader issued has finished before TMEM is released
      if (leader) mma_commit(&sm.mma_drain);
      mbar_wait_teardown(&sm.mma_drain, 0);
    }
  } else {
    // -------------------------------------------------------------- softmax
    const int hb = warp >> 2;                // key-column half [64hb, 64hb + 64) of every tile
    const int wq = warp & 3;                 // TMEM lane quarter of this warp
    const int row = wq * 32 + lane;          // row inside a Q tile
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const float c = p.c_log2;
    uint32_t* err = &g_err_bf16;
    float m_used[kNQ] = {-INFINITY, -INFINITY};
    float l[kNQ] = {0.0f, 0.0f};             // this thread's half of the row sums
    bool ok = true;

    for (int j = 0; j < n && ok; ++j) {
#pragma unroll
      for (int i = 0; i < kNQ; ++i) {
        const uint32_t tS = tmem + lane_off + 128u * i + 64u * hb;
        const uint32_t tO = tmem + lane_off + 256u + 128u * i + 64u * hb;
        if (!mbar_wait_warp(&sm.s_full[i], j & 1, abort_flag, err, kErrTimeoutMma)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t s[64];
        uint32_t(&s0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[0]);
        uint32_t(&s1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[32]);
        tmem_ld32(tS + 0, s0);
        tmem_ld32(tS + 32, s1);
        tmem_ld_wait();
        tmem_reg_fence(s0);
        tmem_reg_fence(s1);
        const int valid = p.S - j * kBN - 64 * hb;   // valid keys in this half (may be <= 0)
        if (valid < 64) {
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (e >= valid) s[e] = f2u(-INFINITY);
        }
        // the row maximum over both halves: publish this half's, read the other's
        const float lm = fmaxf(max32(&s[0]), max32(&s[32]));
        sm.xmax[i][hb][row] = lm;
        __threadfence_block();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.xch[i]);
        if (!mbar_wait_warp(&sm.xch[i], j & 1, abort_flag, err, kErrTimeoutSync)) {
          ok = false;
          break;
        }
        const float m_cand = fmaxf(lm, sm.xmax[i][hb ^ 1][row]) * c;
        // a row whose tile maximum passed its reference by more than kTau moves the
        // reference (both halves of the row decide alike); O and l are brought to
        // the new reference by the factor sc
        const bool need = m_cand > m_used[i] + kTau;
        const float sc = need ? ex2_approx(m_used[i] - m_cand) : 1.0f;
        if (need) {
          l[i] *= sc;
          m_used[i] = m_cand;
        }
        const float neg_m = -m_used[i];
        float rs0 = 0.0f, rs1 = 0.0f;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          // 32 scores -> 16 packed BF16 pairs: P columns [32hb + 16cc, 32hb + 16cc + 16)
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float x0, x1;
            ffma2(x0, x1, u2f(s[32 * cc + 2 * e]), u2f(s[32 * cc + 2 * e + 1]), c, c, neg_m, neg_m);
            const float p0 = ex2_approx(x0);
            const float p1 = ex2_approx(x1);
            fadd2(rs0, rs1, rs0, rs1, p0, p1);
            pk[e] = pack_bf16x2(p0, p1);
          }
          tmem_st16(tmem + lane_off + 128u * i + 32u * hb + 16u * cc, pk);
        }
        l[i] += rs0 + rs1;
        if (j > 0 && __any_sync(0xffffffffu, need)) {
          // O_i must hold P_{j-1} V_{j-1} before this half of its columns is rescaled,
          // and be rescaled before P_j V_j accumulates into it
          if (!mbar_wait_warp(&sm.o_done[i], (j - 1) & 1, abort_flag, err, kErrTimeoutMma)) {
            tmem_st_wait();
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int c2 = 0; c2 < 4; ++c2) {
            uint32_t o[16];
            tmem_ld16(tO + 16 * c2, o);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = f2u(u2f(o[e]) * sc);
            tmem_st16(tO + 16 * c2, o);
          }
        }
        // this warpgroup's half of P_i is in TMEM: the P V MMA on those keys may start
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.p_full[i][hb]);
      }
    }

    // epilogue: both halves' row sums, then this half of O's columns
#pragma unroll
    for (int i = 0; i < kNQ; ++i) {
      if (!ok || n == 0) break;
      if (!mbar_wait_warp(&sm.o_done[i], (n - 1) & 1, abort_flag, err, kErrTimeoutMma)) {
        ok = false;
        break;
      }
      tc_fence_after();
      sm.xsum[i][hb][row] = l[i];
      __threadfence_block();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.xfin[i]);
      if (!mbar_wait_warp(&sm.xfin[i], 0, abort_flag, err, kErrTimeoutSync)) {
        ok = false;
        break;
      }
      const float inv_l = 1.0f / (l[i] + sm.xsum[i][hb ^ 1][row]);
      const int grow = q_row0 + i * kBM + row;
      const uint32_t tO = tmem + lane_off + 256u + 128u * i + 64u * hb;
      __nv_bfloat16* dst =
          p.o + (long long)b * p.o_sb + (long long)grow * p.o_ss + (long long)h * p.o_sh + 64 * hb;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t o[32];
        tmem_ld32(tO + 32 * cc, o);
        tmem_ld_wait();
        tmem_reg_fence(o);
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) w[e] = pack_bf16x2(u2f(o[2 * e]) * inv_l, u2f(o[2 * e + 1]) * inv_l);
        if (grow < p.S) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * cc);
#pragma unroll
          for (int v = 0; v < 4; ++v) d4[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) {
    __syncwarp();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

size_t attn_bf16_smem_bytes() { return sizeof(Smem) + 1024; }

cudaError_t launch_attn_bf16(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                             void* o, long long o_sb, long long o_ss, long long o_sh, int B, int S, int H,
                             float c_log2, cudaStream_t stream) {
  static bool attr_done[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  const size_t smem = attn_bf16_smem_bytes();
  if (!attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attn_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  Params p;
  p.o = reinterpret_cast<__nv_bfloat16*>(o);
  p.o_sb = o_sb;
  p.o_ss = o_ss;
  p.o_sh = o_sh;
  p.S = S;
  p.n_tiles = (S + kBN - 1) / kBN;
  p.c_log2 = c_log2;
  dim3 grid((S + kNQ * kBM - 1) / (kNQ * kBM), H, B);
  attn_bf16_kernel<<<grid, kThreads, smem, stream>>>(tm_q, tm_k, tm_v, p);
  return cudaGetLastError();
}

cudaError_t read_and_clear_err_bf16(uint32_t* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_err_bf16, sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  const uint32_t zero = 0;
  return cudaMemcpyToSymbol(g_err_bf16, &zero, sizeof(uint32_t));
}

}  // namespace sa
