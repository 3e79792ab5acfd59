// Paged grouped-head split-KV decode and the (m, l, o) split merge.
//
// "S12 FlashAttention": 实现 (walk the block table page by page, a page holds
// min(page_size, seq_len - p*page_size) valid tokens), 组合 (block table +
// grouped-head sharing + the (m, l, o) update in one loop), 它还解锁了什么 and
// 练习 1 (flash-decoding: cut the keys across thread blocks, merge the partial
// triples with the recurrence's rescale).
//
// decode_partials_kernel — one warp per (sequence, kv head, split):
//   - the warp's lane 0 streams its split's pages through a kStages-deep ring
//     in shared memory with TMA (K and V page of one kv head: 16 rows x 128
//     bf16 = 4 KB each, 128-byte swizzled so the fragment loads below are
//     bank-conflict free), completion counted on one mbarrier per stage;
//   - the G = H/Hkv query heads that share the kv head are the rows of a
//     16-row mma.sync tile (rows >= G are padding): S = Q K^T for the page is
//     2 n-tiles x 8 k-steps of m16n8k16, P V is 16 n-tiles x 1 k-step;
//   - the online-softmax state (m, l per row, o in the accumulator
//     fragments) is updated per page in the exp2 domain; the guard uses 0 as
//     the reference while a row has seen only masked keys;
//   - tokens past seq_len in the last page are masked in S and their V rows
//     are zeroed in shared memory before P V (0 * NaN would poison O).
//   The warp writes its split's unnormalised triple (m in natural units,
//   l = sum exp(s - m), o = sum exp(s - m) V) to the workspace.
//
// split_combine_kernel — one warp per (sequence, head): M = max m_x,
//   w_x = exp(m_x - M), O = sum w_x o_x / sum w_x l_x, LSE = M + ln l.
//
// Fused form (decode_partials_kernel<true>, "S12 FlashAttention", 接下来: fuse
//   the small-batch decode): the last split of each (sequence, kv head) to
//   finish, found by an atomic ticket (no waiting on other warps), runs the
//   same merge for the group's query heads in the same launch.
//
// decode_gather_kernel — a checking tool for the block-table walk: the
//   decode's units, page ranges, lookups, tensor copies and swizzled page
//   layout, with the gathered K and V rows copied out to dense buffers.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#include "fa_internal.h"
#include "ptx.cuh"
#include "tma_host.h"

namespace fa {
namespace {

constexpr int kPage = 16;           // tokens per page
constexpr int kD = 128;             // head dim (d == dv)
// 4 warps x 2 pages in flight per warp (64 KB of ring per CTA, three CTAs per
// SM): measured best on GB300 for the 64-sequence workload at 4, 8 and 16
// splits (193-195 us, 0.89 of the measured HBM copy bandwidth); 4 x 4 gave
// 209 us, 4 x 3 199 us, 2 x 8 361 us.
constexpr int kWarps = 4;           // units per CTA
constexpr int kMaxRankedSeqs = 256;  // launches with more sequences keep index order
constexpr int kStages = 2;          // pages in flight per warp
constexpr int kHalfBytes = kPage * 64 * 2;     // one 64-column swizzled half page: 2 KB
constexpr int kPageBytes = 2 * kHalfBytes;     // 4 KB (K or V of one page and kv head)
constexpr int kStageBytes = 2 * kPageBytes;    // K + V
constexpr int kSmemBytes = kWarps * kStages * kStageBytes + kWarps * kStages * 8;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// byte offset of (row, 16-byte unit) inside a 128-byte-swizzled 64-column half
__device__ __forceinline__ uint32_t swz(int row, int unit) {
  return (uint32_t)(row * 128 + ((unit ^ (row & 7)) << 4));
}

__device__ __forceinline__ void issue_page(const CUtensorMap* tmK, const CUtensorMap* tmV,
                                           uint32_t stage_base, uint32_t bar, int phys, int Hkv,
                                           int g) {
  const int row = (phys * Hkv + g) * kPage;
  ptx::mbar_arrive_expect_tx(bar, kStageBytes);
  ptx::tma_load_2d(stage_base, tmK, 0, row, bar);
  ptx::tma_load_2d(stage_base + kHalfBytes, tmK, 64, row, bar);
  ptx::tma_load_2d(stage_base + kPageBytes, tmV, 0, row, bar);
  ptx::tma_load_2d(stage_base + kPageBytes + kHalfBytes, tmV, 64, row, bar);
}

__device__ __forceinline__ int page_id(const int* bt_row, int p, int num_pages, bool& bad) {
  int id = __ldg(bt_row + p);
  bad = id < 0 || id >= num_pages;
  return bad ? 0 : id;
}

// A sequence length outside [0, max_blocks * 16] would walk past its row of
// the block table: it is recorded (FA_ERR_INVALID_ARG) and the sequence is
// treated as empty.
__device__ __forceinline__ int checked_len(int L, int max_blocks, int* status, int lane) {
  if (L >= 0 && (long long)L <= (long long)max_blocks * kPage) return L;
  if (lane == 0) atomicExch(status, kDevInvalidArg);
  return 0;
}

// Pages [pb, pe) of split x of X over a sequence of L tokens: page-aligned,
// near-equal, ceil(x P / X) .. ceil((x + 1) P / X) for P = ceil(L / 16).
__device__ __forceinline__ void split_pages(int x, int X, int L, int& pb, int& pe) {
  const int P = L > 0 ? (L + kPage - 1) / kPage : 0;
  pb = (int)(((long long)x * P + X - 1) / X);
  pe = (int)(((long long)(x + 1) * P + X - 1) / X);
}

// How the merge reads partials: through the read-only cache (the separate
// merge kernel, whose partials were written by an earlier launch), or from L2
// (the fused path, which reads partials other SMs wrote during the same
// launch, after a fence).
struct LoadReadOnly {
  __device__ float operator()(const float* a) const { return __ldg(a); }
  __device__ float4 v4(const float* a) const { return __ldg(reinterpret_cast<const float4*>(a)); }
};
struct LoadL2 {
  __device__ float operator()(const float* a) const { return __ldcg(a); }
  __device__ float4 v4(const float* a) const { return __ldcg(reinterpret_cast<const float4*>(a)); }
};

// Merge of the X split triples of one (sequence, head) t by one warp: M = max
// m_x, w_x = exp(m_x - M) (0 for an empty split), O = sum w_x o_x / sum w_x
// l_x, LSE = M + ln l.  The same arithmetic for either load policy, so the
// separate and the fused merge give identical bits.
template <typename Load>
__device__ __forceinline__ void merge_splits(const float* __restrict__ part_m,
                                             const float* __restrict__ part_l,
                                             const float* __restrict__ part_o,
                                             __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                                             size_t t, int X, int dv, int lane, Load load) {
  const float* pm = part_m + t * X;
  const float* pl = part_l + t * X;
  // lane x holds split x and x + 32 (X <= 64): the weights are computed once
  // and handed out by shuffles, so the o loads below are all independent
  const float m0 = lane < X ? load(pm + lane) : -INFINITY;
  const float m1 = lane + 32 < X ? load(pm + lane + 32) : -INFINITY;
  float M = fmaxf(m0, m1);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  __nv_bfloat16* orow = o + t * dv;
  if (M == -INFINITY) {
    for (int c = lane * 4; c < dv; c += 128) {
      *reinterpret_cast<uint2*>(orow + c) = make_uint2(0u, 0u);
    }
    if (lane == 0 && lse != nullptr) lse[t] = -INFINITY;
    return;
  }
  const float w0 = m0 == -INFINITY ? 0.f : exp2f((m0 - M) * kLog2e);
  const float w1 = m1 == -INFINITY ? 0.f : exp2f((m1 - M) * kLog2e);
  float l = (lane < X ? w0 * load(pl + lane) : 0.f) + (lane + 32 < X ? w1 * load(pl + lane + 32) : 0.f);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const float* po = part_o + t * X * dv;
  // every lane runs every chunk (the shuffles need the whole warp); lanes
  // past dv load and store nothing
  for (int c0 = 0; c0 < dv; c0 += 128) {
    const int c = c0 + lane * 4;
    const bool active = c < dv;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int x0 = 0; x0 < X; x0 += 8) {
      float4 v[8];
      float w[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int x = x0 + u;
        w[u] = __shfl_sync(0xffffffffu, x < 32 ? w0 : w1, x & 31);
        v[u] = active && x < X ? load.v4(po + (size_t)x * dv + c) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        acc.x = fmaf(w[u], v[u].x, acc.x);
        acc.y = fmaf(w[u], v[u].y, acc.y);
        acc.z = fmaf(w[u], v[u].z, acc.z);
        acc.w = fmaf(w[u], v[u].w, acc.w);
      }
    }
    if (active) {
      uint2 packed;
      packed.x = ptx::pack_bf16x2(acc.x * inv, acc.y * inv);
      packed.y = ptx::pack_bf16x2(acc.z * inv, acc.w * inv);
      *reinterpret_cast<uint2*>(orow + c) = packed;
    }
  }
  if (lane == 0 && lse != nullptr) lse[t] = l > 0.f ? M + logf(l) : -INFINITY;
}

// FUSED: after writing its triple, the warp takes a ticket of its (sequence,
// kv head); the split that takes the last one merges the X triples of the G
// query heads (merge_splits) and writes O and LSE, so no second launch is
// needed.  Every unit takes its ticket, the timed-out ones included, and the
// merging split sets the count back to 0 for the next call.
template <bool FUSED>
__global__ void __launch_bounds__(kWarps * 32)
decode_partials_kernel(const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const __nv_bfloat16* __restrict__ q, const int* __restrict__ block_table,
                       const int* __restrict__ seq_lens, int num_seqs, int H, int Hkv,
                       int num_pages, int max_blocks, int X, float scale_log2,
                       float* __restrict__ part_m, float* __restrict__ part_l,
                       float* __restrict__ part_o, int* status, int skip_first_copy,
                       int* __restrict__ tickets, __nv_bfloat16* __restrict__ o,
                       float* __restrict__ lse) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int unit = blockIdx.x * kWarps + warp;
  // Longest sequences first: CTAs start in block order, so a grid whose
  // heavy units come last ends on a long tail.  With few sequences every CTA
  // ranks them by length (ties by index) in shared memory; unit u then
  // belongs to the (u / (X * Hkv))-th longest.
  __shared__ int s_len[kMaxRankedSeqs];
  __shared__ int s_order[kMaxRankedSeqs];
  const bool ranked = num_seqs <= kMaxRankedSeqs;
  if (ranked) {
    for (int t = threadIdx.x; t < num_seqs; t += blockDim.x) s_len[t] = seq_lens[t];
    __syncthreads();
    for (int t = threadIdx.x; t < num_seqs; t += blockDim.x) {
      const int Lt = s_len[t];
      int rank = 0;
      for (int u = 0; u < num_seqs; ++u) rank += (s_len[u] > Lt) || (s_len[u] == Lt && u < t);
      s_order[rank] = t;
    }
    __syncthreads();
  }
  // the merge launched behind this kernel may start once every CTA of this
  // one is running (it waits for this kernel's completion before reading)
  asm volatile("griddepcontrol.launch_dependents;");
  if (unit >= num_seqs * Hkv * X) return;

  const int x = unit % X;
  const int g = (unit / X) % Hkv;
  const int s = ranked ? s_order[unit / (X * Hkv)] : unit / (X * Hkv);
  const int G = H / Hkv;
  const int L = checked_len(seq_lens[s], max_blocks, status, lane);
  int pb, pe;
  split_pages(x, X, L, pb, pe);
  const int* bt_row = block_table + (size_t)s * max_blocks;

  const uint32_t ring = ptx::smem_u32(smem + warp * kStages * kStageBytes);
  const uint32_t bars = ptx::smem_u32(smem + kWarps * kStages * kStageBytes) + warp * kStages * 8;

  if (lane == 0) {
    for (int st = 0; st < kStages; ++st) ptx::mbar_init(bars + 8 * st, 1);
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
    ptx::prefetch_tmap(&tmK);
    ptx::prefetch_tmap(&tmV);
    for (int it = 0; it < kStages && pb + it < pe; ++it) {
      // test hook: with skip_first_copy the first page is never requested, so
      // its wait runs out and the timeout path (status, drain, return) runs
      if (skip_first_copy && it == 0) continue;
      bool bad;
      int id = page_id(bt_row, pb + it, num_pages, bad);
      if (bad) atomicExch(status, kDevBadBlockTable);
      issue_page(&tmK, &tmV, ring + it * kStageBytes, bars + 8 * it, id, Hkv, g);
    }
  }
  __syncwarp();

  // Q fragments (A operand, rows = query heads of the group, zero padding)
  const int r0 = lane >> 2;        // fragment row
  const int c2 = (lane & 3) * 2;   // fragment column pair
  uint32_t qa[kD / 16][4];
  {
    const uint32_t* q0 = reinterpret_cast<const uint32_t*>(q + ((size_t)s * H + g * G + r0) * kD);
    const uint32_t* q1 = reinterpret_cast<const uint32_t*>(q + ((size_t)s * H + g * G + r0 + 8) * kD);
    const bool v0 = r0 < G, v1 = r0 + 8 < G;
#pragma unroll
    for (int t = 0; t < kD / 16; ++t) {
      qa[t][0] = v0 ? __ldg(q0 + (16 * t + c2) / 2) : 0u;
      qa[t][1] = v1 ? __ldg(q1 + (16 * t + c2) / 2) : 0u;
      qa[t][2] = v0 ? __ldg(q0 + (16 * t + 8 + c2) / 2) : 0u;
      qa[t][3] = v1 ? __ldg(q1 + (16 * t + 8 + c2) / 2) : 0u;
    }
  }

  float oacc[kD / 8][4];
#pragma unroll
  for (int j = 0; j < kD / 8; ++j) oacc[j][0] = oacc[j][1] = oacc[j][2] = oacc[j][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  bool timed_out = false;
  int p_fail = 0;

  // ldmatrix lane roles
  const int mi = lane >> 3;   // which 8x8 matrix this lane addresses
  const int rr = lane & 7;    // row inside it

  for (int p = pb; p < pe; ++p) {
    const int it = p - pb;
    const int st = it % kStages;
    const uint32_t kbase = ring + st * kStageBytes;
    const uint32_t vbase = kbase + kPageBytes;
    if (!ptx::mbar_wait(bars + 8 * st, (it / kStages) & 1, status)) {
      timed_out = true;
      p_fail = p;
      break;
    }
    bool bad;
    page_id(bt_row, p, num_pages, bad);
    int nvalid = min(kPage, L - p * kPage);
    if (bad) nvalid = 0;
    if (nvalid < kPage) {
      // zero the V rows of the tokens past the end (16 units of 16 B per row)
      uint8_t* vgen = smem + (vbase - ptx::smem_u32(smem));
      for (int idx = lane; idx < (kPage - nvalid) * 16; idx += 32) {
        int row = nvalid + idx / 16, u = idx % 16;
        *reinterpret_cast<uint4*>(vgen + (u / 8) * kHalfBytes + swz(row, u % 8)) =
            make_uint4(0u, 0u, 0u, 0u);
      }
      __syncwarp();
    }

    // S = Q K^T for the page: n-tile 0 = tokens 0-7, n-tile 1 = tokens 8-15
    float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int t = 0; t < kD / 16; ++t) {
      const int half = t >> 2;
      const int u0 = (t & 3) * 2;
      const int tok = rr + ((mi >> 1) << 3);
      const int unitx = u0 + (mi & 1);
      uint32_t b0, b1, b2, b3;
      ptx::ldmatrix_x4(kbase + half * kHalfBytes + swz(tok, unitx), b0, b1, b2, b3);
      ptx::mma_bf16_16816(sacc[0], qa[t], b0, b1);
      ptx::mma_bf16_16816(sacc[1], qa[t], b2, b3);
    }

    // online softmax update (rows r0 and r0+8), exp2 domain
    float pv[2][4];
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int tok = nt * 8 + c2 + (e & 1);
        const float sv = tok < nvalid ? sacc[nt][e] * scale_log2 : -INFINITY;
        pv[nt][e] = sv;
        mx[e >> 1] = fmaxf(mx[e >> 1], sv);
      }
    float alpha[2], ref[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 1));
      mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 2));
      const float m_new = fmaxf(m_run[hr], mx[hr]);
      ref[hr] = m_new == -INFINITY ? 0.f : m_new;
      alpha[hr] = m_run[hr] == -INFINITY ? 1.f : ptx::ex2(m_run[hr] - ref[hr]);
      m_run[hr] = m_new;
      l_run[hr] *= alpha[hr];
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float pe_ = ptx::ex2(pv[nt][e] - ref[e >> 1]);
        pv[nt][e] = pe_;
        l_run[e >> 1] += pe_;
      }
#pragma unroll
    for (int j = 0; j < kD / 8; ++j) {
      oacc[j][0] *= alpha[0];
      oacc[j][1] *= alpha[0];
      oacc[j][2] *= alpha[1];
      oacc[j][3] *= alpha[1];
    }
    uint32_t pa[4];
    pa[0] = ptx::pack_bf16x2(pv[0][0], pv[0][1]);
    pa[1] = ptx::pack_bf16x2(pv[0][2], pv[0][3]);
    pa[2] = ptx::pack_bf16x2(pv[1][0], pv[1][1]);
    pa[3] = ptx::pack_bf16x2(pv[1][2], pv[1][3]);

    // O += P V: pairs of n-tiles (16 dv columns) per ldmatrix.x4.trans
#pragma unroll
    for (int jj = 0; jj < kD / 16; ++jj) {
      const int half = jj >> 2;
      const int u0 = (jj & 3) * 2;
      const int tok = rr + ((mi & 1) << 3);
      const int unitx = u0 + (mi >> 1);
      uint32_t b0, b1, b2, b3;
      ptx::ldmatrix_x4_trans(vbase + half * kHalfBytes + swz(tok, unitx), b0, b1, b2, b3);
      ptx::mma_bf16_16816(oacc[2 * jj], pa, b0, b1);
      ptx::mma_bf16_16816(oacc[2 * jj + 1], pa, b2, b3);
    }
    __syncwarp();

    // refill this stage with the page kStages ahead
    if (lane == 0 && p + kStages < pe) {
      ptx::fence_proxy_async_smem();
      bool bad2;
      int id = page_id(bt_row, p + kStages, num_pages, bad2);
      if (bad2) atomicExch(status, kDevBadBlockTable);
      issue_page(&tmK, &tmV, kbase, bars + 8 * st, id, Hkv, g);
    }
  }

  if (timed_out) {
    // Let the copies already in flight (pages [p_fail, p_fail + kStages)) land
    // before the warp's shared memory is released; each wait is bounded too.
    if (lane == 0) {
      for (int pp = p_fail + 1; pp < min(pe, p_fail + kStages); ++pp) {
        const int it = pp - pb;
        ptx::mbar_wait(bars + 8 * (it % kStages), (it / kStages) & 1, nullptr);
      }
    }
    __syncwarp();
    if (!FUSED) return;
  } else {
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 1);
      l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 2);
    }
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int r = r0 + hr * 8;
      if (r >= G) continue;
      const size_t idx = ((size_t)s * H + g * G + r) * X + x;
      if (!FA_IN_BOUNDS(idx, (size_t)num_seqs * H * X, status)) continue;
      if ((lane & 3) == 0) {
        part_m[idx] = m_run[hr] == -INFINITY ? -INFINITY : m_run[hr] * kLn2;
        part_l[idx] = l_run[hr];
      }
      float* orow = part_o + idx * kD;
#pragma unroll
      for (int j = 0; j < kD / 8; ++j)
        *reinterpret_cast<float2*>(orow + j * 8 + c2) =
            make_float2(oacc[j][hr * 2], oacc[j][hr * 2 + 1]);
    }
  }
  if constexpr (FUSED) {
    // The warp barrier orders every lane's triple stores before lane 0's
    // ticket; the ticket is a release (this triple) and an acquire (the
    // other splits' triples, for the unit that merges) at device scope; the
    // second barrier passes the acquire on to the other lanes' loads.
    __syncwarp();
    int ticket = 0;
    if (lane == 0) ticket = ptx::atom_add_acq_rel_gpu(tickets + (size_t)s * Hkv + g, 1);
    ticket = __shfl_sync(0xffffffffu, ticket, 0);
    __syncwarp();
    if (ticket == X - 1) {
      for (int r = 0; r < G; ++r)
        merge_splits(part_m, part_l, part_o, o, lse, (size_t)s * H + g * G + r, X, kD, lane,
                     LoadL2());
      if (lane == 0) tickets[(size_t)s * Hkv + g] = 0;   // ready for the next call
    }
  }
}

__global__ void __launch_bounds__(128)
split_combine_kernel(const float* __restrict__ part_m, const float* __restrict__ part_l,
                     const float* __restrict__ part_o, __nv_bfloat16* __restrict__ o,
                     float* __restrict__ lse, int pairs, int X, int dv) {
  // Launched right behind the partials kernel as a programmatic dependent, the
  // merge's blocks may start during that kernel's tail: wait here until it
  // has completed and its partials are visible (at once without a predecessor).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int t = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= pairs) return;
  merge_splits(part_m, part_l, part_o, o, lse, (size_t)t, X, dv, lane, LoadReadOnly());
}

// Block-table check: the decode's units (one warp per sequence, kv head and
// split, in index order), each walking its split's pages with the decode's
// range rule (split_pages), lookups (page_id) and tensor copies (issue_page)
// into the same 128-byte-swizzled page layout, then copying the valid rows out
// of shared memory (swz) to dense K and V buffers [num_seqs][max_blocks * 16]
// [Hkv][128]: token t of sequence s lands on row s * max_blocks * 16 + t.
// Rows at or past seq_len are not written.  One page in flight per warp.
constexpr int kGatherSmemBytes = kWarps * kStageBytes + kWarps * 8 + 1024;  // + alignment slack

__global__ void __launch_bounds__(kWarps * 32)
decode_gather_kernel(const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const int* __restrict__ block_table,
                     const int* __restrict__ seq_lens, int num_seqs, int Hkv, int num_pages,
                     int max_blocks, int X, __nv_bfloat16* __restrict__ k_out,
                     __nv_bfloat16* __restrict__ v_out, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int unit = blockIdx.x * kWarps + warp;
  if (unit >= num_seqs * Hkv * X) return;
  const int x = unit % X;
  const int g = (unit / X) % Hkv;
  const int s = unit / (X * Hkv);
  const int L = checked_len(seq_lens[s], max_blocks, status, lane);
  int pb, pe;
  split_pages(x, X, L, pb, pe);
  const int* bt_row = block_table + (size_t)s * max_blocks;
  const uint8_t* stage = smem + warp * kStageBytes;
  const uint32_t stage_a = ptx::smem_u32(stage);
  const uint32_t bar = ptx::smem_u32(smem + kWarps * kStageBytes) + warp * 8;
  if (lane == 0) {
    ptx::mbar_init(bar, 1);
    ptx::fence_mbar_init();
  }
  __syncwarp();
  const size_t row0 = (size_t)s * max_blocks * kPage;
  for (int p = pb; p < pe; ++p) {
    bool bad;
    const int id = page_id(bt_row, p, num_pages, bad);
    if (lane == 0) {
      if (bad) atomicExch(status, kDevBadBlockTable);
      ptx::fence_proxy_async_smem();   // the previous page's reads come before this copy
      issue_page(&tmK, &tmV, stage_a, bar, id, Hkv, g);
    }
    if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar, (p - pb) & 1, status))) {
      // the copy may still land: let it (bounded) before the warp leaves
      if (lane == 0) ptx::mbar_wait(bar, (p - pb) & 1, nullptr);
      __syncwarp();
      return;
    }
    const int nvalid = bad ? 0 : min(kPage, L - p * kPage);
    // 16-byte units: K rows then V rows, 16 units (two swizzled halves) per row
    for (int idx = lane; idx < 2 * nvalid * 16; idx += 32) {
      const int which = idx / (nvalid * 16);
      const int rem = idx - which * nvalid * 16;
      const int row = rem >> 4, u = rem & 15;
      const uint4 val = *reinterpret_cast<const uint4*>(stage + which * kPageBytes +
                                                        (u >> 3) * kHalfBytes + swz(row, u & 7));
      __nv_bfloat16* out = which ? v_out : k_out;
      const size_t orow = (row0 + (size_t)p * kPage + row) * Hkv + g;
      if (FA_IN_BOUNDS(orow, (size_t)num_seqs * max_blocks * kPage * Hkv, status))
        *reinterpret_cast<uint4*>(out + orow * kD + u * 8) = val;
    }
    __syncwarp();
  }
}

// Failure-detection test hook: FA_TEST_FORCE_WAIT_TIMEOUT=1 in the
// environment makes every decode warp skip its first page copy, so its
// bounded wait expires (after ~1 s), FA_ERR_TIMEOUT is recorded and the warp
// returns without writing its partials.  Unset in normal use.
int skip_first_copy_for_tests() {
  const char* v = getenv("FA_TEST_FORCE_WAIT_TIMEOUT");
  return (v != nullptr && v[0] == '1') ? 1 : 0;
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream, bool fused) {
  if (p.num_seqs == 0) return cudaSuccess;
  CUtensorMap tmK, tmV;
  const uint64_t rows = (uint64_t)p.num_pages * p.Hkv * kPage;
  const uint64_t dims[2] = {(uint64_t)kD, rows};
  const uint64_t strides[1] = {(uint64_t)kD * 2};
  const uint32_t box[2] = {64, (uint32_t)kPage};
  if (!make_tmap_bf16(&tmK, p.k_cache, 2, dims, strides, box) ||
      !make_tmap_bf16(&tmV, p.v_cache, 2, dims, strides, box))
    return cudaErrorInvalidValue;
  auto kernel = fused ? decode_partials_kernel<true> : decode_partials_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return e;
  const int units = p.num_seqs * p.Hkv * p.num_splits;
  const int grid = (units + kWarps - 1) / kWarps;
  kernel<<<grid, kWarps * 32, kSmemBytes, stream>>>(
      tmK, tmV, static_cast<const __nv_bfloat16*>(p.q), p.block_table, p.seq_lens, p.num_seqs,
      p.H, p.Hkv, p.num_pages, p.max_blocks, p.num_splits, p.scale * kLog2e, p.part_m, p.part_l,
      p.part_o, p.status, skip_first_copy_for_tests(), p.tickets,
      static_cast<__nv_bfloat16*>(p.o), p.lse);
  return cudaGetLastError();
}

cudaError_t launch_decode_partials(const DecodeParams& p, cudaStream_t stream) {
  return launch_decode(p, stream, false);
}

cudaError_t launch_decode_gather(const GatherParams& p, cudaStream_t stream) {
  if (p.num_seqs == 0) return cudaSuccess;
  CUtensorMap tmK, tmV;
  const uint64_t rows = (uint64_t)p.num_pages * p.Hkv * kPage;
  const uint64_t dims[2] = {(uint64_t)kD, rows};
  const uint64_t strides[1] = {(uint64_t)kD * 2};
  const uint32_t box[2] = {64, (uint32_t)kPage};
  if (!make_tmap_bf16(&tmK, p.k_cache, 2, dims, strides, box) ||
      !make_tmap_bf16(&tmV, p.v_cache, 2, dims, strides, box))
    return cudaErrorInvalidValue;
  const int units = p.num_seqs * p.Hkv * p.num_splits;
  const int grid = (units + kWarps - 1) / kWarps;
  decode_gather_kernel<<<grid, kWarps * 32, kGatherSmemBytes, stream>>>(
      tmK, tmV, p.block_table, p.seq_lens, p.num_seqs, p.Hkv, p.num_pages, p.max_blocks,
      p.num_splits, static_cast<__nv_bfloat16*>(p.k_out), static_cast<__nv_bfloat16*>(p.v_out),
      p.status);
  return cudaGetLastError();
}

cudaError_t launch_split_combine(const CombineParams& p, cudaStream_t stream, bool behind_partials) {
  const int pairs = p.num_seqs * p.H;
  if (pairs == 0) return cudaSuccess;
  if (!behind_partials) {
    split_combine_kernel<<<(pairs + 3) / 4, 128, 0, stream>>>(
        p.part_m, p.part_l, p.part_o, static_cast<__nv_bfloat16*>(p.o), p.lse, pairs,
        p.num_splits, p.dv);
    return cudaGetLastError();
  }
  // programmatic dependent launch: the merge's launch overlaps the partials
  // kernel's tail instead of starting after it has drained
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((pairs + 3) / 4));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, split_combine_kernel, p.part_m, p.part_l, p.part_o,
                            static_cast<__nv_bfloat16*>(p.o), p.lse, pairs, p.num_splits, p.dv);
}

}  // namespace fa
