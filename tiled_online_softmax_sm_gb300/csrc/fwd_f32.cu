// fp32 attention forward on the CUDA cores (IEEE fp32 arithmetic, no TF32).
//
// The online-softmax recurrence of "手搓 Attention" §7 (version 4) and
// "S12 FlashAttention" (解法), one CTA per (batch, head, block of query rows):
//   - the CTA keeps its query rows in registers and streams K/V tiles of
//     kTileN rows through shared memory, one tile live at a time;
//   - kThreadsPerRow lanes share a query row; each owns d/kThreadsPerRow of
//     the dimensions (for Q·K) and dv/kThreadsPerRow (for the accumulator),
//     interleaved in float4 chunks so that the lanes of a row read adjacent
//     16-byte words of a K/V row;
//   - per tile: raw dot products q·k_j carried as compensated pairs, tile
//     max, m_new, the rescale alpha = exp(scale·(m - m_new)) and
//     p_j = exp(scale·(s_j - m_new)), both evaluated as 2^(x·log2 e); whole
//     tiles above the causal diagonal are skipped and a fully masked tile uses
//     0 as its reference (the -inf/NaN guard of "S12 FlashAttention", 实现).
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "fa_internal.h"

namespace fa {
namespace {

// Lanes of a warp sharing a query row.  The kernel is bound by latency (a
// 256-row problem is only 256 rows): measured on GB300 at n = m = 256, d = 64,
// 4 lanes 92 us, 8 lanes 66 us, 16 lanes 60 us per launch.
constexpr int kThreadsPerRow = 16;
// Key groups of a CTA: the CTA's key tiles are dealt to its groups (tile t to
// group t % kGroups), each with its own copy of the rows' state and its own
// tile buffer, and the groups' (max, sum, acc) are merged at the end the way
// split partials are ("S12 FlashAttention", 它还解锁了什么): a row's key tiles
// run side by side.  The kernel is bound by latency, so more and smaller CTAs
// with more groups finish sooner: at n = m = 256, d = 64, groups of 128
// threads x 4 took 21.3 us, groups of 64 x 8 took 11.8 us (GB300).  Eight
// groups of d = dv = 128 tiles would need 256 KB of shared memory, so that
// instance keeps 128 x 4.
template <int D, int DV>
struct Shape {
  static constexpr bool kSmall = D + DV <= 192;
  static constexpr int kGroupThreads = kSmall ? 64 : 128;           // one key group
  static constexpr int kGroups = kSmall ? 8 : 4;
  static constexpr int kRowsPerCta = kGroupThreads / kThreadsPerRow;  // query rows per CTA
  static constexpr int kThreads = kGroupThreads * kGroups;
};

// bar.sync on the named barrier of one group (count: the group's threads)
__device__ __forceinline__ void group_sync(int group, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + group), "r"(count) : "memory");
}
constexpr int kTileN = 32;                      // keys per K/V tile
constexpr float kLog2e = 1.4426950408889634f;

// Error-free transformations (Knuth's TwoSum; TwoProduct with one FMA) used
// to carry each score as an unevaluated pair hi + lo.  With scores in the
// hundreds a single fp32 score holds only ~1e-5 absolute precision, which the
// weights exp(s - m) would inherit; the pair keeps s - m accurate to fp32
// relative precision of the difference itself.  The __f*_rn intrinsics are
// never contracted into FMAs, which would break the transformations.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float z = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, z)), __fsub_rn(b, z));
}

__device__ __forceinline__ void dot2_step(float a, float b, float& hi, float& lo) {
  const float p = __fmul_rn(a, b);
  const float r = fmaf(a, b, -p);  // exact: a*b = p + r
  float s, e;
  two_sum(hi, p, s, e);
  hi = s;
  lo = __fadd_rn(lo, __fadd_rn(e, r));
}

__device__ __forceinline__ void pair_add(float& hi, float& lo, float hi2, float lo2) {
  float s, e;
  two_sum(hi, hi2, s, e);
  hi = s;
  lo = __fadd_rn(__fadd_rn(lo, lo2), e);
}

// (a_hi + a_lo) - (b_hi + b_lo), scaled, in fp32
__device__ __forceinline__ float pair_diff_scaled(float a_hi, float a_lo, float b_hi, float b_lo,
                                                  float scale) {
  return __fmul_rn(__fadd_rn(__fsub_rn(a_hi, b_hi), __fsub_rn(a_lo, b_lo)), scale);
}

template <int D, int DV>
__global__ void __launch_bounds__(Shape<D, DV>::kThreads)
fwd_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
               const float* __restrict__ v, float* __restrict__ o, float* __restrict__ lse,
               int B, int H, int Hkv, int n, int m, float scale, int causal, int* status) {
  using S = Shape<D, DV>;
  extern __shared__ float4 smem4[];
  const int group = threadIdx.x / S::kGroupThreads;
  const int tid = threadIdx.x % S::kGroupThreads;   // thread within its group
  float4* sK = smem4 + group * kTileN * ((D + DV) / 4);   // [kTileN][D/4] of this group
  float4* sV = sK + kTileN * (D / 4);                     // [kTileN][DV/4]

  const float scale_log2 = scale * kLog2e;
  const int row = tid / kThreadsPerRow;
  const int part = tid % kThreadsPerRow;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int hk = h / (H / Hkv);
  const int q0 = blockIdx.x * S::kRowsPerCta;
  const int i = q0 + row;                       // query index of this row
  const bool row_valid = i < n;

  constexpr int QC = D / (4 * kThreadsPerRow);    // float4 chunks of q owned by this thread
  constexpr int VC = DV / (4 * kThreadsPerRow);   // float4 chunks of acc owned by this thread
  static_assert(QC >= 1 && VC >= 1, "a thread owns at least one float4 of q and of acc");

  float4 qr[QC];
  float4 acc[VC];
  {
    const float4* qrow = reinterpret_cast<const float4*>(q + (((size_t)b * n + (row_valid ? i : 0)) * H + h) * D);
#pragma unroll
    for (int c = 0; c < QC; ++c)
      qr[c] = row_valid ? qrow[c * kThreadsPerRow + part] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int c = 0; c < VC; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // running maximum of the raw dot products, as a pair; -inf until a key is seen
  float m_hi = -INFINITY, m_lo = 0.f;
  float l_run = 0.f;

  int kv_end = m;
  const int off = m - n;  // causal, bottom-right: query i sees keys j <= i + off
  if (causal) kv_end = min(m, q0 + S::kRowsPerCta + off);
  const size_t k_row_stride = (size_t)Hkv * D;
  const size_t v_row_stride = (size_t)Hkv * DV;
  const float* kbase = k + ((size_t)b * m * Hkv + hk) * D;
  const float* vbase = v + ((size_t)b * m * Hkv + hk) * DV;

  for (int j0 = group * kTileN; j0 < kv_end; j0 += S::kGroups * kTileN) {
    const int cols = min(kTileN, m - j0);
    group_sync(group, S::kGroupThreads);  // previous tile fully consumed
    for (int idx = tid; idx < kTileN * (D / 4); idx += S::kGroupThreads) {
      int r = idx / (D / 4), c = idx % (D / 4);
      sK[idx] = r < cols ? reinterpret_cast<const float4*>(kbase + (size_t)(j0 + r) * k_row_stride)[c]
                         : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int idx = tid; idx < kTileN * (DV / 4); idx += S::kGroupThreads) {
      int r = idx / (DV / 4), c = idx % (DV / 4);
      sV[idx] = r < cols ? reinterpret_cast<const float4*>(vbase + (size_t)(j0 + r) * v_row_stride)[c]
                         : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    group_sync(group, S::kGroupThreads);

    int vis = cols;                 // visible keys of this row in the tile: [0, vis)
    if (causal) vis = min(vis, i + off - j0 + 1);
    if (!row_valid) vis = 0;

    float s_hi[kTileN], s_lo[kTileN];
    float t_hi = -INFINITY, t_lo = 0.f;   // tile maximum
#pragma unroll
    for (int j = 0; j < kTileN; ++j) {
      const float4* kr = sK + j * (D / 4);
      float hi = 0.f, lo = 0.f;
#pragma unroll
      for (int c = 0; c < QC; ++c) {
        const float4 kk = kr[c * kThreadsPerRow + part];
        dot2_step(qr[c].x, kk.x, hi, lo);
        dot2_step(qr[c].y, kk.y, hi, lo);
        dot2_step(qr[c].z, kk.z, hi, lo);
        dot2_step(qr[c].w, kk.w, hi, lo);
      }
#pragma unroll
      for (int off = 1; off < kThreadsPerRow; off <<= 1)
        pair_add(hi, lo, __shfl_xor_sync(0xffffffffu, hi, off), __shfl_xor_sync(0xffffffffu, lo, off));
      if (j >= vis) {
        hi = -INFINITY;
        lo = 0.f;
      }
      s_hi[j] = hi;
      s_lo[j] = lo;
      if (hi > t_hi) {
        t_hi = hi;
        t_lo = lo;
      }
    }
    // m_new = max(m, tile max); reference 0 while nothing is visible (guard)
    float n_hi = m_hi, n_lo = m_lo;
    if (t_hi > n_hi) {
      n_hi = t_hi;
      n_lo = t_lo;
    }
    const bool empty = n_hi == -INFINITY;
    const float r_hi = empty ? 0.f : n_hi, r_lo = empty ? 0.f : n_lo;
    const float alpha = m_hi == -INFINITY ? 1.f : exp2f(pair_diff_scaled(m_hi, m_lo, r_hi, r_lo, scale_log2));
#pragma unroll
    for (int c = 0; c < VC; ++c) {
      acc[c].x *= alpha; acc[c].y *= alpha; acc[c].z *= alpha; acc[c].w *= alpha;
    }
    float psum = 0.f;
#pragma unroll
    for (int j = 0; j < kTileN; ++j) {
      const float p = s_hi[j] == -INFINITY ? 0.f
                                           : exp2f(pair_diff_scaled(s_hi[j], s_lo[j], r_hi, r_lo, scale_log2));
      psum += p;
      const float4* vr = sV + j * (DV / 4);
#pragma unroll
      for (int c = 0; c < VC; ++c) {
        const float4 vv = vr[c * kThreadsPerRow + part];
        acc[c].x = fmaf(p, vv.x, acc[c].x);
        acc[c].y = fmaf(p, vv.y, acc[c].y);
        acc[c].z = fmaf(p, vv.z, acc[c].z);
        acc[c].w = fmaf(p, vv.w, acc[c].w);
      }
    }
    l_run = l_run * alpha + psum;
    m_hi = n_hi;
    m_lo = n_lo;
  }

  // ---- merge the groups: each publishes (max pair, sum, acc) of its rows;
  // group 0 rescales them to the common max and adds them up
  __syncthreads();   // every group is done with its tile buffer
  float* st = reinterpret_cast<float*>(smem4);   // [S::kGroups][S::kRowsPerCta][4 + DV]
  constexpr int kRowFloats = 4 + DV;   // max pair, sum, a pad word: acc stays 16-byte aligned
  float* mine = st + (group * S::kRowsPerCta + row) * kRowFloats;
  if (part == 0) {
    mine[0] = m_hi;
    mine[1] = m_lo;
    mine[2] = l_run;
  }
#pragma unroll
  for (int c = 0; c < VC; ++c)
    reinterpret_cast<float4*>(mine + 4)[c * kThreadsPerRow + part] = acc[c];
  __syncthreads();
  if (group != 0) return;
  float g_hi = -INFINITY, g_lo = 0.f;   // max over the groups
  for (int g = 0; g < S::kGroups; ++g) {
    const float* o_g = st + (g * S::kRowsPerCta + row) * kRowFloats;
    if (o_g[0] > g_hi) {
      g_hi = o_g[0];
      g_lo = o_g[1];
    }
  }
  l_run = 0.f;
#pragma unroll
  for (int c = 0; c < VC; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (g_hi != -INFINITY) {
    for (int g = 0; g < S::kGroups; ++g) {
      const float* o_g = st + (g * S::kRowsPerCta + row) * kRowFloats;
      if (o_g[0] == -INFINITY) continue;   // this group saw no key of the row
      const float w = exp2f(pair_diff_scaled(o_g[0], o_g[1], g_hi, g_lo, scale_log2));
      l_run = fmaf(w, o_g[2], l_run);
#pragma unroll
      for (int c = 0; c < VC; ++c) {
        const float4 a = reinterpret_cast<const float4*>(o_g + 4)[c * kThreadsPerRow + part];
        acc[c].x = fmaf(w, a.x, acc[c].x);
        acc[c].y = fmaf(w, a.y, acc[c].y);
        acc[c].z = fmaf(w, a.z, acc[c].z);
        acc[c].w = fmaf(w, a.w, acc[c].w);
      }
    }
  }
  m_hi = g_hi;
  m_lo = g_lo;

  if (!row_valid) return;
  const size_t oi = ((size_t)b * n + i) * H + h;   // O has B * n * H rows of DV
  if (!FA_IN_BOUNDS(oi, (size_t)B * n * H, status)) return;
  const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
  float4* orow = reinterpret_cast<float4*>(o + oi * DV);
#pragma unroll
  for (int c = 0; c < VC; ++c) {
    const float4 x = acc[c];
    orow[c * kThreadsPerRow + part] = make_float4(x.x * inv, x.y * inv, x.z * inv, x.w * inv);
  }
  if (lse != nullptr && part == 0)
    lse[((size_t)b * H + h) * n + i] =
        l_run > 0.f ? (m_hi + m_lo) * scale + logf(l_run) : -INFINITY;
}

template <int D, int DV>
cudaError_t launch(const FwdParams& p, cudaStream_t stream) {
  using S = Shape<D, DV>;
  const size_t tiles = sizeof(float) * kTileN * (D + DV) * S::kGroups;
  const size_t merge = sizeof(float) * S::kGroups * S::kRowsPerCta * (4 + DV);
  const size_t smem = tiles > merge ? tiles : merge;
  cudaError_t e = cudaFuncSetAttribute(fwd_f32_kernel<D, DV>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((p.n + S::kRowsPerCta - 1) / S::kRowsPerCta, p.H, p.B);
  fwd_f32_kernel<D, DV><<<grid, S::kThreads, smem, stream>>>(
      static_cast<const float*>(p.q), static_cast<const float*>(p.k),
      static_cast<const float*>(p.v), static_cast<float*>(p.o), p.lse, p.B, p.H, p.Hkv, p.n,
      p.m, p.scale, p.causal, p.status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_f32(const FwdParams& p, cudaStream_t stream) {
  if (p.n == 0 || p.B == 0) return cudaSuccess;
  if (p.d == 64 && p.dv == 64) return launch<64, 64>(p, stream);
  if (p.d == 64 && p.dv == 128) return launch<64, 128>(p, stream);
  if (p.d == 128 && p.dv == 64) return launch<128, 64>(p, stream);
  if (p.d == 128 && p.dv == 128) return launch<128, 128>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
