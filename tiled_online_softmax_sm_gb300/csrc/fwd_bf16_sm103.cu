// bf16 attention forward for sm_103a on the tcgen05 tensor cores.
//
// The tiled online-softmax recurrence ("手搓 Attention" §7 version 4; "S12
// FlashAttention", 解法) with the loop order of "FlashAttention推理优化实战100例
// 01" (a CTA owns query tiles and streams every K/V tile past them), mapped to
// Blackwell:
//
//   CTA = two 128-row query tiles of one (batch, head), 12 warps:
//     warp 0      TMA producer: Q tiles once, then K(j), V(j) through a
//                 kStages-slot shared-memory ring (128-byte swizzle)
//     warp 1      owns the tensor memory (512 columns) and, on one lane,
//                 issues every tcgen05.mma:
//                   S_i = Q_i K(j)^T   (SS: both operands in shared memory)
//                   O_i += P_i V(j)    (TS: P in tensor memory, V MN-major)
//     warps 2-3   idle (they complete the first warpgroup)
//     warps 4-7   softmax for query tile 0, warps 8-11 for tile 1: thread =
//                 one query row = one tensor-memory lane, so row max and row
//                 sum need no shuffles.
//   Tensor memory: S_0 | S_1 (128 fp32 columns each), O_0 | O_1 (d columns
//   each).  P_i (bf16) overwrites the first 64 columns of S_i; the next
//   S_i MMA is issued after the P_i V MMA, and tcgen05 MMAs of one thread
//   execute in issue order.
//
// Per K/V tile a softmax thread loads its S row, masks (causal diagonal tile,
// keys past the sequence end), takes the row max in log2 units
// (s * scale * log2 e), and forms p = 2^(s - ref).  The reference ref is the
// running max, raised only when a tile's max exceeds it by more than 8 (a
// factor 256): then acc (O in tensor memory) and l are multiplied by
// alpha = 2^(m_old - m_new) before the next P V.  Between raises p can reach
// 256, which bf16 and fp32 hold exactly enough; the final O = acc / l and
// LSE = (ref + log2 l) ln 2 are exact in any case.  While a row has seen only
// masked keys its reference is 0, so exp(-inf - -inf) never occurs ("S12
// FlashAttention", 实现).  Whole K/V tiles above the causal diagonal are never
// loaded or multiplied ("手搓 Attention" §6).
//
// Every mbarrier wait is bounded; on a timeout the CTA records it in the
// device status word, stops issuing work, lets copies in flight land and
// frees its tensor memory.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "fa_internal.h"
#include "ptx.cuh"
#include "tma_host.h"

namespace fa {
namespace {

constexpr int kBlockM = 128;   // query rows per tile (= tensor-memory lanes)
constexpr int kBlockN = 128;   // keys per K/V tile
constexpr int kThreads = 384;  // 12 warps = 3 warpgroups
// Register split (setmaxnreg): the launch gives every thread kLaunchRegs; the
// TMA/MMA warpgroup drops to kProducerRegs and the two softmax warpgroups rise
// to kSoftmaxRegs.  128*(kProducerRegs + 2*kSoftmaxRegs) must not exceed
// 384*kLaunchRegs, or the increase would wait forever; the build refuses a
// library whose kernel does not use exactly kLaunchRegs registers.
constexpr int kLaunchRegs = 168;
constexpr int kProducerRegs = 72;
constexpr int kSoftmaxRegs = 216;
static_assert(128 * (kProducerRegs + 2 * kSoftmaxRegs) <= kThreads * kLaunchRegs, "register split");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct Cfg {
  static constexpr int kChunks = D / 64;                 // 64-column swizzle chunks
  static constexpr int kTileBytes = 128 * D * 2;         // Q, K or V tile
  static constexpr int kStages = D == 128 ? 4 : 8;       // K/V ring slots
  static constexpr int kQBytes = 2 * kTileBytes;
  static constexpr int kSmem = kQBytes + kStages * kTileBytes + 1024;  // + alignment slack
  static constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(128, kBlockN, false, false);
  static constexpr uint32_t kIdescO = ptx::idesc_bf16_f32(128, D, false, true);
};

struct Shared {
  uint64_t q_full[2];
  uint64_t s_full[2];
  uint64_t p_full[4];   // [tile][half]
  uint64_t o_done[2];
  uint64_t kv_full[8];
  uint64_t kv_empty[8];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, __nv_bfloat16* __restrict__ o,
                float* __restrict__ lse, const int* __restrict__ cu_q,
                const int* __restrict__ cu_k, int H, int Hkv, int n, int m, int total_q,
                int total_k, int num_pairs, float scale_log2, int causal, int lse_stride_h,
                int lse_stride_b, int* status) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Shared sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work unit: (batch b, head h, pair t of query tiles); heaviest pairs first
  const int bh = blockIdx.x;
  const int h = bh % H;
  const int b = bh / H;
  const int t = num_pairs - 1 - (int)blockIdx.y;
  const int hk = h / (H / Hkv);
  int q_len = n, kv_len = m, q_row0 = b * n, k_row0 = b * m;
  if (cu_q != nullptr) {
    q_row0 = __ldg(cu_q + b);
    q_len = __ldg(cu_q + b + 1) - q_row0;
    k_row0 = __ldg(cu_k + b);
    kv_len = __ldg(cu_k + b + 1) - k_row0;
    if (q_row0 < 0 || q_len < 0 || q_row0 + q_len > total_q || k_row0 < 0 || kv_len < 0 ||
        k_row0 + kv_len > total_k) {
      if (threadIdx.x == 0) atomicExch(status, kDevInvalidArg);
      return;  // offsets outside the buffers: skip the sequence, touch nothing
    }
  }
  const int q_start0 = t * 2 * kBlockM;
  if (q_start0 >= q_len) return;  // whole CTA idle (uniform exit before any barrier)
  int n_kv[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int qs = q_start0 + i * kBlockM;
    int keys = kv_len;
    if (causal) keys = min(kv_len, qs + kBlockM);
    n_kv[i] = (qs >= q_len || keys <= 0) ? 0 : (keys + kBlockN - 1) / kBlockN;
  }
  const int n_kv_max = max(n_kv[0], n_kv[1]);

  uint8_t* sQ = smem;                        // [2][kChunks][128 rows][128 B]
  uint8_t* sKV = smem + C::kQBytes;          // [kStages][kChunks][128 rows][128 B]

  const uint32_t bar_q = ptx::smem_u32(&sh.q_full[0]);
  const uint32_t bar_s = ptx::smem_u32(&sh.s_full[0]);
  const uint32_t bar_p = ptx::smem_u32(&sh.p_full[0]);
  const uint32_t bar_o = ptx::smem_u32(&sh.o_done[0]);
  const uint32_t bar_kvf = ptx::smem_u32(&sh.kv_full[0]);
  const uint32_t bar_kve = ptx::smem_u32(&sh.kv_empty[0]);
  const uint32_t bar_drain = ptx::smem_u32(&sh.drain);
  volatile int* abort_flag = &sh.abort;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(bar_q + 8 * i, 1);
      ptx::mbar_init(bar_s + 8 * i, 1);
      ptx::mbar_init(bar_p + 16 * i, kBlockM);
      ptx::mbar_init(bar_p + 16 * i + 8, kBlockM);
      ptx::mbar_init(bar_o + 8 * i, 1);
    }
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(bar_kvf + 8 * s, 1);
      ptx::mbar_init(bar_kve + 8 * s, 1);
    }
    ptx::mbar_init(bar_drain, 1);
    sh.abort = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(&sh.tmem_base), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tbase = sh.tmem_base;

  if (warp < 4) {
  ptx::setmaxnreg_dec<kProducerRegs>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ptx::prefetch_tmap(&tmQ);
      ptx::prefetch_tmap(&tmK);
      ptx::prefetch_tmap(&tmV);
      for (int i = 0; i < 2; ++i) {
        if (n_kv[i] == 0) continue;
        const uint32_t dst = ptx::smem_u32(sQ + i * C::kTileBytes);
        ptx::mbar_arrive_expect_tx(bar_q + 8 * i, C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          ptx::tma_load_3d(dst + c * 16384, &tmQ, 64 * c, h, q_row0 + q_start0 + i * kBlockM,
                           bar_q + 8 * i);
      }
      int issued = 0;
      bool ok = true;
      for (int j = 0; j < n_kv_max && ok; ++j) {
        for (int which = 0; which < 2; ++which) {  // K then V
          const int li = 2 * j + which;
          const int slot = li % C::kStages;
          if (!ptx::mbar_wait(bar_kve + 8 * slot, ((li / C::kStages) & 1) ^ 1, status, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t dst = ptx::smem_u32(sKV + slot * C::kTileBytes);
          ptx::mbar_arrive_expect_tx(bar_kvf + 8 * slot, C::kTileBytes);
          const CUtensorMap* map = which == 0 ? &tmK : &tmV;
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
            ptx::tma_load_3d(dst + c * 16384, map, 64 * c, hk, k_row0 + j * kBlockN,
                             bar_kvf + 8 * slot);
          issued = li + 1;
        }
      }
      if (!ok) {
        // let the last loads of every slot land before shared memory is released
        for (int li = max(0, issued - C::kStages); li < issued; ++li)
          ptx::mbar_wait(bar_kvf + 8 * (li % C::kStages), (li / C::kStages) & 1, nullptr);
        for (int i = 0; i < 2; ++i)
          if (n_kv[i] > 0) ptx::mbar_wait(bar_q + 8 * i, 0, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = true;
      for (int i = 0; i < 2 && ok; ++i)
        if (n_kv[i] > 0) ok = ptx::mbar_wait(bar_q + 8 * i, 0, status, abort_flag);
      const uint32_t q_addr[2] = {ptx::smem_u32(sQ), ptx::smem_u32(sQ + C::kTileBytes)};
      auto issue_s = [&](int i, int slot) {
        const uint32_t kaddr = ptx::smem_u32(sKV + slot * C::kTileBytes);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
          const uint64_t ad = ptx::smem_desc_sw128(q_addr[i] + off, 16, 1024);
          const uint64_t bd = ptx::smem_desc_sw128(kaddr + off, 16, 1024);
          ptx::mma_ss(tbase + i * kBlockN, ad, bd, C::kIdescS, k > 0);
        }
      };
      // O_i += P_i V(j) in two halves of 64 keys, each issued once the softmax
      // warps have stored that half of P; false if a wait failed
      auto issue_pv = [&](int i, int slot, int j) -> bool {
        const uint32_t vaddr = ptx::smem_u32(sKV + slot * C::kTileBytes);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          if (!ptx::mbar_wait(bar_p + 16 * i + 8 * hf, j & 1, status, abort_flag)) return false;
          ptx::tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kBlockN / 32; ++kk) {
            const int k = hf * (kBlockN / 32) + kk;
            const uint64_t bd = ptx::smem_desc_sw128(vaddr + k * 2048, 16384, 1024);
            ptx::mma_ts(tbase + 256 + i * D, tbase + i * kBlockN + k * 8, bd, C::kIdescO,
                        (j > 0 || k > 0) ? 1u : 0u);
          }
        }
        return true;
      };
      // prologue: S_i(0)
      if (ok && n_kv_max > 0) {
        ok = ptx::mbar_wait(bar_kvf, 0, status, abort_flag);
        if (ok) {
          ptx::tc_fence_after();
          for (int i = 0; i < 2; ++i) {
            if (n_kv[i] == 0) continue;
            issue_s(i, 0);
            ptx::tc_commit(bar_s + 8 * i);
          }
          ptx::tc_commit(bar_kve);  // K(0) slot
        }
      }
      for (int j = 0; j < n_kv_max && ok; ++j) {
        const int lv = 2 * j + 1, sv = lv % C::kStages;
        const int lk = 2 * j + 2, sk = lk % C::kStages;
        const bool has_next = j + 1 < n_kv_max;
        if (!(ok = ptx::mbar_wait(bar_kvf + 8 * sv, (lv / C::kStages) & 1, status, abort_flag))) break;
        if (j < n_kv[0]) {
          if (!(ok = issue_pv(0, sv, j))) break;
          if (j == n_kv[0] - 1) ptx::tc_commit(bar_o);
        }
        if (has_next) {
          if (!(ok = ptx::mbar_wait(bar_kvf + 8 * sk, (lk / C::kStages) & 1, status, abort_flag))) break;
          ptx::tc_fence_after();
        }
        if (j + 1 < n_kv[0]) {
          issue_s(0, sk);
          ptx::tc_commit(bar_s);
        }
        if (j < n_kv[1]) {
          if (!(ok = issue_pv(1, sv, j))) break;
          if (j == n_kv[1] - 1) ptx::tc_commit(bar_o + 8);
        }
        ptx::tc_commit(bar_kve + 8 * sv);  // V(j) slot
        if (j + 1 < n_kv[1]) {
          issue_s(1, sk);
          ptx::tc_commit(bar_s + 8);
        }
        if (has_next) ptx::tc_commit(bar_kve + 8 * sk);  // K(j+1) slot
      }
      // no tcgen05.mma may still run when the tensor memory is released
      ptx::tc_commit(bar_drain);
      ptx::mbar_wait(bar_drain, 0, nullptr);
    }
  }
  } else {
    ptx::setmaxnreg_inc<kSoftmaxRegs>();
    // ------------------------------------------------------------ softmax
    const int i = (warp - 4) / 4;             // query tile of this warpgroup
    const int quarter = warp & 3;             // tensor-memory lane quarter
    const int r = quarter * 32 + lane;        // row in the tile
    const int q_start = q_start0 + i * kBlockM;
    const int qi = q_start + r;               // query index in the sequence
    const uint32_t lane_base = tbase + ((uint32_t)(quarter * 32) << 16);
    const uint32_t s_col = lane_base + i * kBlockN;
    const uint32_t o_col = lane_base + 256 + i * D;
    float m_ref = -INFINITY;   // running reference (log2 units)
    float l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv[i]; ++j) {
      // warp-uniform outcome: the tcgen05.ld/st below are warp-collective
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar_s + 8 * i, j & 1, status, abort_flag));
      if (!ok) break;
      ptx::tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) ptx::tmem_ld32(s_col + c * 32, sr[c]);
      ptx::tmem_wait_ld();
      // mask: keys past the end, and the causal diagonal (only the last tile of a row)
      const int k0 = j * kBlockN;
      if (j == n_kv[i] - 1) {
        int vis = kv_len - k0;
        if (causal) vis = min(vis, qi - k0 + 1);
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (c * 32 + e >= vis) sr[c][e] = __float_as_uint(-INFINITY);
      }
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          mx = ptx::fmax3(mx, __uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1]));
      const float m_tile = mx * scale_log2;    // scale > 0: max commutes with it
      const bool raise = m_tile > m_ref + kRescaleThreshold || (m_ref == -INFINITY && m_tile > -INFINITY);
      float alpha = 1.f;
      if (raise) {
        alpha = m_ref == -INFINITY ? 1.f : ptx::ex2(m_ref - m_tile);
        m_ref = m_tile;
        l_run *= alpha;
      }
      const float ref = m_ref == -INFINITY ? 0.f : m_ref;
      // rescale acc first when this warp raised a reference after the first
      // tile: no P V of this tile may run before it
      if (__any_sync(0xffffffffu, raise && j > 0 && alpha != 1.f)) {
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          ptx::tmem_ld32(o_col + c * 32, ov);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
          ptx::tmem_st32(o_col + c * 32, ov);
        }
      }
      // p = 2^(s*scale*log2e - ref), two halves of 64 keys; each half is
      // handed to the MMA warp as soon as it sits in tensor memory
      const uint64_t sc2 = ptx::f2_bits(scale_log2, scale_log2);
      const uint64_t nref2 = ptx::f2_bits(-ref, -ref);
      uint64_t lsum2 = ptx::f2_bits(0.f, 0.f);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t pr[32];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c = hf * 2 + cc;
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const uint64_t x = ptx::ffma2(
                ptx::f2_bits(__uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1])), sc2, nref2);
            float x0, x1;
            ptx::f2_split(x, x0, x1);
            const float p0 = ptx::ex2(x0);
            const float p1 = ptx::ex2(x1);
            lsum2 = ptx::fadd2(lsum2, ptx::f2_bits(p0, p1));
            pr[cc * 16 + e / 2] = ptx::pack_bf16x2(p0, p1);
          }
        }
        ptx::tmem_st32(s_col + hf * 32, pr);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar_p + 16 * i + 8 * hf);
      }
      float ls0, ls1;
      ptx::f2_split(lsum2, ls0, ls1);
      l_run += ls0 + ls1;
    }

    // ---- epilogue: O = acc / l (bf16), LSE = (ref + log2 l) ln 2
    const bool row_valid = qi < q_len;
    const size_t orow = (size_t)(q_row0 + qi) * H + h;
    if (ok && n_kv[i] > 0) {
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar_o + 8 * i, 0, status, abort_flag));
      ptx::tc_fence_after();
    }
    if (ok) {
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(o + orow * D);
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        if (n_kv[i] > 0) {  // warp-uniform: every lane loads, only valid rows store
          ptx::tmem_ld32(o_col + c * 32, ov);
          ptx::tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = 0u;
        }
        if (row_valid) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 w;
            w.x = ptx::pack_bf16x2(__uint_as_float(ov[8 * u + 0]) * inv, __uint_as_float(ov[8 * u + 1]) * inv);
            w.y = ptx::pack_bf16x2(__uint_as_float(ov[8 * u + 2]) * inv, __uint_as_float(ov[8 * u + 3]) * inv);
            w.z = ptx::pack_bf16x2(__uint_as_float(ov[8 * u + 4]) * inv, __uint_as_float(ov[8 * u + 5]) * inv);
            w.w = ptx::pack_bf16x2(__uint_as_float(ov[8 * u + 6]) * inv, __uint_as_float(ov[8 * u + 7]) * inv);
            dst[c * 4 + u] = w;
          }
        }
      }
      if (row_valid && lse != nullptr)
        lse[(size_t)b * lse_stride_b + (size_t)h * lse_stride_h + (q_row0 - (cu_q ? 0 : b * n)) + qi] =
            l_run > 0.f ? (m_ref + __log2f(l_run)) * kLn2 : -INFINITY;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tbase, 512);
  }
}

template <int D>
cudaError_t launch(const FwdParams& p, cudaStream_t stream, const char** why) {
  using C = Cfg<D>;
  const bool varlen = p.cu_q != nullptr;
  // 3-D views (dim, head, token row) of Q, K, V; out-of-range rows read as 0.
  const uint64_t q_rows = varlen ? (uint64_t)(p.total_q > 0 ? p.total_q : 1) : (uint64_t)p.B * p.n;
  const uint64_t k_rows = varlen ? (uint64_t)(p.total_k > 0 ? p.total_k : 1) : (uint64_t)p.B * p.m;
  CUtensorMap tq, tk, tv;
  const uint32_t box[3] = {64, 1, 128};
  {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)p.H, q_rows};
    const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)p.H * D * 2};
    if (!make_tmap_bf16(&tq, p.q, 3, dims, strides, box)) {
      *why = "tensor map for q";
      return cudaErrorInvalidValue;
    }
  }
  {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)p.Hkv, k_rows > 0 ? k_rows : 1};
    const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)p.Hkv * D * 2};
    if (!make_tmap_bf16(&tk, p.m > 0 ? p.k : p.q, 3, dims, strides, box) ||
        !make_tmap_bf16(&tv, p.m > 0 ? p.v : p.q, 3, dims, strides, box)) {
      *why = "tensor map for k/v";
      return cudaErrorInvalidValue;
    }
  }
  cudaError_t e = cudaFuncSetAttribute(fwd_bf16_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) {
    *why = "cudaFuncSetAttribute(fwd_bf16)";
    return e;
  }
  const int num_pairs = (p.n + 2 * kBlockM - 1) / (2 * kBlockM);
  dim3 grid(p.B * p.H, num_pairs);
  // LSE layout: dense [B][H][n] ; varlen [H][Tq]
  const int lse_stride_h = varlen ? p.total_q : p.n;
  const int lse_stride_b = varlen ? 0 : p.H * p.n;
  const float scale_log2 = p.scale * kLog2e;
  fwd_bf16_kernel<D><<<grid, kThreads, C::kSmem, stream>>>(
      tq, tk, tv, static_cast<__nv_bfloat16*>(p.o), p.lse, p.cu_q, p.cu_k, p.H, p.Hkv, p.n, p.m,
      varlen ? p.total_q : p.B * p.n, varlen ? p.total_k : p.B * p.m, num_pairs, scale_log2,
      p.causal, lse_stride_h, lse_stride_b, p.status);
  e = cudaGetLastError();
  if (e != cudaSuccess) *why = "fwd_bf16 launch";
  return e;
}

}  // namespace

cudaError_t launch_fwd_bf16(const FwdParams& p, cudaStream_t stream, const char** why) {
  if (p.d == 128 && p.dv == 128) return launch<128>(p, stream, why);
  if (p.d == 64 && p.dv == 64) return launch<64>(p, stream, why);
  *why = "fwd_bf16: unsupported head dim";
  return cudaErrorInvalidValue;
}

}  // namespace fa
