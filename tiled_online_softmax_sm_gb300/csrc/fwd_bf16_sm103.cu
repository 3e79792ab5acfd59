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
//   each; at d = 64 in bf16, 80 columns at 128-column spacing, the last 16
//   holding l_p).  P_i (bf16) overwrites the first 64 columns of S_i; the next
//   S_i MMA is issued after the P_i V MMA, and tcgen05 MMAs of one thread
//   execute in issue order.
//
// Per K/V tile a softmax thread loads its S row, masks (causal diagonal tile,
// keys past the sequence end) and forms p = 2^(s - ref) in log2 units
// (s * scale * log2 e).  The reference ref is the running max, raised only
// when a tile's max exceeds it by more than 8 (a factor 256): then acc (O in
// tensor memory) and l are multiplied by alpha = 2^(m_old - m_new) before the
// next P V.  Between raises p can reach 256, inside bf16's and fp32's range.
// Two row sums are kept: l of the exact p, for LSE = (ref + log2 l) ln 2, and
// l_p of the bf16-rounded p the P V MMA multiplies, for O = acc / l_p, so that
// O is a weighted mean of V rows whose weights sum to one whatever the
// rounding (a row one key dominates gets that key's V row back).  At d = 64
// the tensor core forms l_p itself, as extra columns of the P V product with
// a block of ones; at d = 128 the softmax threads add up the packed P.  The row max
// itself is taken only when needed: p is first formed
// against the current ref, and a tile row sum of at most 256 proves no raise
// is due (see the softmax loop).  While a row has seen only
// masked keys its reference is 0, so exp(-inf - -inf) never occurs ("S12
// FlashAttention", 实现).  Whole K/V tiles above the causal diagonal are never
// loaded or multiplied ("手搓 Attention" §6).  Causal is aligned bottom-right:
// query i of n sees keys j <= i + (m - n) (top-left when n == m).
//
// Dense non-causal launches whose last wave of pair units would leave at
// least half the CTAs idle run those units as split units instead: one query
// tile whose K/V tiles are halved between the two softmax warpgroups, the two
// (m, l, O) states merged at the end inside the CTA with the same rescale
// ("S12 FlashAttention", 练习 1), so the last wave takes about half as long.
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
constexpr int kProducerRegs = 88;
constexpr int kSoftmaxRegs = 208;
static_assert(128 * (kProducerRegs + 2 * kSoftmaxRegs) <= kThreads * kLaunchRegs, "register split");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// The reference is raised only when a tile's max passes it by more than the
// threshold (log2 units), so p stays at most 2^8: e4m3 P saturates at 448.
// For bf16, O is divided by the sum of the same rounded p, so its accuracy
// does not depend on the threshold; 12, 16 and 24 measured the same speed.
constexpr float kRescaleThreshold = 8.0f;
constexpr float kRaiseSum = 256.0f;   // 2^kRescaleThreshold

// Tile geometry for head dim D and operand type (bf16, or e4m3 with FP8).
template <int D, bool FP8 = false>
struct Cfg {
  static constexpr int kElem = FP8 ? 1 : 2;                 // bytes per element
  static constexpr int kRowBytes = D * kElem;
  static constexpr int kChunkElems = 128 / kElem;           // elements per 128-byte swizzle chunk
  static constexpr int kChunks = kRowBytes / 128;           // chunks per row
  static constexpr int kKStep = 32 / kElem;                 // reduction length of one MMA (32 bytes)
  static constexpr int kTileBytes = 128 * kRowBytes;        // Q, K or V tile
  // bf16 at d = 64: the P V MMA is 16 columns wider than V, and its B operand
  // reads those columns from a block of ones that sits right behind the V
  // tile in every ring slot, so O's accumulator carries l_p (the sum of the
  // bf16 P it multiplied) in columns D .. D+15, accumulated and rescaled by
  // the tensor core with O.  (At d = 128 the tensor memory has no room left.)
  static constexpr bool kOnes = D == 64 && !FP8;
  static constexpr int kSlotBytes = kOnes ? 2 * kTileBytes : kTileBytes;  // ring slot stride
  static constexpr int kStages = kOnes ? 5 : kTileBytes == 32768 ? 4 : 8;  // K/V ring slots
  static constexpr int kON = kOnes ? D + 16 : D;           // O accumulator columns
  static constexpr int kOStride = kOnes ? 128 : D;         // tensor-memory columns between O_0 and O_1
  static constexpr int kQBytes = 2 * kTileBytes;
  static constexpr int kSmem = kQBytes + kStages * kSlotBytes + 1024;  // + alignment slack
  static constexpr uint32_t kIdescS = FP8 ? ptx::idesc_e4m3_f32(128, kBlockN, false, false)
                                          : ptx::idesc_bf16_f32(128, kBlockN, false, false);
  static constexpr uint32_t kIdescO = FP8 ? ptx::idesc_e4m3_f32(128, D, false, true)
                                          : ptx::idesc_bf16_f32(128, kON, false, true);
};

// Varlen and paged launches with at most this many (sequence, query pair)
// combinations get a persistent grid over a heaviest-first list of them.
constexpr int kMaxSortedCombos = 512;

struct Shared {
  uint16_t work[kMaxSortedCombos];    // K/V tiles of combination b * num_pairs + t
  uint16_t order[kMaxSortedCombos];   // combinations, heaviest first
  int n_order;                        // combinations with any work
  uint64_t q_full[2];
  uint64_t q_empty[2];  // Q_i free for the next unit's load
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done[2];
  uint64_t o_empty[2];  // O_i read by the epilogue; the next unit may overwrite it
  uint64_t kv_full[8];
  uint64_t kv_empty[8];
  uint64_t drain;
  uint64_t fix;         // paged: a V tile that reaches past the end, before zeroing
  uint64_t merge_full;  // split unit: warpgroup 1's row states are in mstat
  uint64_t merge_empty; // split unit: warpgroup 0 has read them
  float mstat[kBlockM][3];  // split unit: (m, l, l_p) of each row of warpgroup 1
  uint32_t tmem_base;
  int abort;
};

// One work unit: a pair of 128-row query tiles of one (sequence, head).
// A split unit (dense, the last partial wave only) is one query tile whose
// K/V tiles are halved between the two softmax warpgroups: both Q slots hold
// the same rows, tile 1 starts at K/V tile kv_first[1], and warpgroup 0 merges
// the two (m, l, O) states at the end, reading O_1 from tensor memory.
struct Unit {
  int b, h, hk;
  int q_len, kv_len, q_row0, k_row0, q_start0;
  int q_start[2];  // first query row (in the sequence) of each tile
  int kv_first[2]; // first K/V tile of each tile
  int n_kv[2];     // K/V tiles each query tile needs (0: tile inactive)
  bool rows;       // the unit holds at least one valid query row
  bool bad;        // varlen offsets outside the buffers
  bool split;      // the two tiles are one query tile over two key ranges
};

// Row max of a 128-key S row: 8 independent chains of three-input max (one
// chain would put 64 dependent instructions on the critical path), then a
// small tree.
__device__ __forceinline__ float row_max(const uint32_t (&sr)[4][32]) {
  float mxs[8];
#pragma unroll
  for (int a = 0; a < 8; ++a) mxs[a] = -INFINITY;
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      const int a = (c * 16 + e / 2) & 7;
      mxs[a] = ptx::fmax3(mxs[a], __uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1]));
    }
  return ptx::fmax3(ptx::fmax3(mxs[0], mxs[1], mxs[2]), ptx::fmax3(mxs[3], mxs[4], mxs[5]),
                    fmaxf(mxs[6], mxs[7]));
}

// One softmax row of a tile: p = 2^(s * scale_log2 - ref) for the 128 keys in
// sr (nref2 holds -ref twice), written over the row's S columns as bf16 (2 per
// tensor-memory column) or e4m3 (4 per column), with no wait for the stores.
// Returns the row sum of p.
template <bool FP8>
__device__ __forceinline__ float exp_pass(const uint32_t (&sr)[4][32], uint32_t s_col,
                                          uint64_t sc2, uint64_t nref2) {
  uint64_t lsum2[4];   // four independent packed partial sums
#pragma unroll
  for (int a = 0; a < 4; ++a) lsum2[a] = ptx::f2_bits(0.f, 0.f);
#pragma unroll
  for (int c = 0; c < 4; ++c) {   // keys 32c..32c+31
    uint32_t pr[16];
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      const uint64_t x = ptx::ffma2(
          ptx::f2_bits(__uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1])), sc2, nref2);
      float x0, x1;
      ptx::f2_split(x, x0, x1);
      const float p0 = ptx::ex2(x0);
      const float p1 = ptx::ex2(x1);
      lsum2[(e / 2) & 3] = ptx::fadd2(lsum2[(e / 2) & 3], ptx::f2_bits(p0, p1));
      if constexpr (FP8) {
        const uint32_t h = ptx::pack_e4m3x2(p0, p1);   // keys e, e+1 in the low 16 bits
        if ((e & 2) == 0) pr[e / 4] = h;
        else pr[e / 4] |= h << 16;
      } else {
        pr[e / 2] = ptx::pack_bf16x2(p0, p1);
      }
    }
    if constexpr (FP8) {
      uint32_t p8[8];
#pragma unroll
      for (int w = 0; w < 8; ++w) p8[w] = pr[w];
      ptx::tmem_st8(s_col + c * 8, p8);
    } else {
      ptx::tmem_st16(s_col + c * 16, pr);
    }
  }
  float ls0, ls1;
  ptx::f2_split(ptx::fadd2(ptx::fadd2(lsum2[0], lsum2[1]), ptx::fadd2(lsum2[2], lsum2[3])), ls0, ls1);
  return ls0 + ls1;
}

// bf16 form of the pass above: p = 2^(s * scale_log2 - ref) for the 128 keys
// of sr, packed to bf16 pairs in pp (pp[w] holds keys 2w, 2w+1, key 2w in the
// low half: the row's 64 P columns in tensor-memory order).  With STORE each
// chunk of 32 keys goes to tensor memory as soon as it is packed; otherwise the
// caller stores pp (or discards it).  Returns the row sum of the unrounded p.
template <bool STORE>
__device__ __forceinline__ float exp_pack_bf16(const uint32_t (&sr)[4][32], uint32_t s_col,
                                               uint64_t sc2, uint64_t nref2, uint32_t (&pp)[64]) {
  uint64_t lsum2[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) lsum2[a] = ptx::f2_bits(0.f, 0.f);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      const uint64_t x = ptx::ffma2(
          ptx::f2_bits(__uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1])), sc2, nref2);
      float x0, x1;
      ptx::f2_split(x, x0, x1);
      const float p0 = ptx::ex2(x0);
      const float p1 = ptx::ex2(x1);
      lsum2[(e / 2) & 3] = ptx::fadd2(lsum2[(e / 2) & 3], ptx::f2_bits(p0, p1));
      pp[c * 16 + e / 2] = ptx::pack_bf16x2(p0, p1);
    }
    if constexpr (STORE) {
      uint32_t chunk[16];
#pragma unroll
      for (int w = 0; w < 16; ++w) chunk[w] = pp[c * 16 + w];
      ptx::tmem_st16(s_col + c * 16, chunk);
    }
  }
  float ls0, ls1;
  ptx::f2_split(ptx::fadd2(ptx::fadd2(lsum2[0], lsum2[1]), ptx::fadd2(lsum2[2], lsum2[3])), ls0, ls1);
  return ls0 + ls1;
}

// Row sum of the bf16 P the P V MMA multiplies, in fp32: each bf16 value is
// added to an fp32 accumulator by one mixed-precision add (exact widening,
// one rounding), eight independent chains.
__device__ __forceinline__ float sum_packed_bf16(const uint32_t (&pp)[64]) {
  float acc[8];
#pragma unroll
  for (int a = 0; a < 8; ++a) acc[a] = 0.f;
#pragma unroll
  for (int w = 0; w < 64; ++w) ptx::add_bf16x2_to_f32(acc[2 * (w & 3)], acc[2 * (w & 3) + 1], pp[w]);
  return ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
}

// The unit of query pair t (rows 256t .. 256t+255) of sequence b, head h.
__device__ __forceinline__ Unit make_unit(int b, int h, int t, int H, int Hkv, int n, int m,
                                          int causal, const int* cu_q, const int* cu_k,
                                          int total_q, int total_k, const int* seq_lens,
                                          int max_blocks) {
  Unit U;
  U.h = h;
  U.b = b;
  U.hk = U.h / (H / Hkv);
  U.q_len = n;
  U.kv_len = m;
  U.q_row0 = U.b * n;
  U.k_row0 = U.b * m;
  U.bad = false;
  if (seq_lens != nullptr) {  // paged: keys through the block table
    U.q_row0 = __ldg(cu_q + U.b);
    U.q_len = __ldg(cu_q + U.b + 1) - U.q_row0;
    U.k_row0 = 0;
    U.kv_len = __ldg(seq_lens + U.b);
    U.bad = U.q_row0 < 0 || U.q_len < 0 || U.q_row0 + U.q_len > total_q || U.kv_len < 0 ||
            (long long)U.kv_len > (long long)max_blocks * 16;   // wide: max_blocks may pass 2^27
  } else if (cu_q != nullptr) {
    U.q_row0 = __ldg(cu_q + U.b);
    U.q_len = __ldg(cu_q + U.b + 1) - U.q_row0;
    U.k_row0 = __ldg(cu_k + U.b);
    U.kv_len = __ldg(cu_k + U.b + 1) - U.k_row0;
    U.bad = U.q_row0 < 0 || U.q_len < 0 || U.q_row0 + U.q_len > total_q || U.k_row0 < 0 ||
            U.kv_len < 0 || U.k_row0 + U.kv_len > total_k;
  }
  U.q_start0 = t * 2 * kBlockM;
  U.rows = !U.bad && U.q_start0 < U.q_len;
  U.split = false;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int qs = U.q_start0 + i * kBlockM;
    U.q_start[i] = qs;
    U.kv_first[i] = 0;
    int keys = U.kv_len;   // causal: the tile's last row sees keys < qs + 128 + (m - n)
    if (causal) keys = min(U.kv_len, qs + kBlockM + (U.kv_len - U.q_len));
    U.n_kv[i] = (!U.rows || qs >= U.q_len || keys <= 0) ? 0 : (keys + kBlockN - 1) / kBlockN;
  }
  return U;
}

// Query tile `tile` of the pair unit R as a split unit: its K/V tiles halved
// between the two warpgroups.  A query tile with one K/V tile stays a plain
// one-tile unit (tile 1 inactive).
__device__ __forceinline__ Unit split_unit(Unit R, int tile) {
  Unit U = R;
  // selects, not R.x[tile]: a runtime index would put the unit in local memory
  const int n = tile == 0 ? R.n_kv[0] : R.n_kv[1];
  const int qs = tile == 0 ? R.q_start[0] : R.q_start[1];
  const int half = (n + 1) / 2;
  U.q_start[0] = U.q_start[1] = qs;
  U.q_start0 = qs;
  U.rows = R.rows && n > 0;
  U.n_kv[0] = half;
  U.n_kv[1] = n - half;
  U.kv_first[0] = 0;
  U.kv_first[1] = half;
  U.split = U.n_kv[1] > 0;
  return U;
}

// PAGED: K and V come from page caches [pages][Hkv][16][d] through the block
// table (2-D tensor maps, one 16-row box per page), seq_lens gives each
// sequence's key count; otherwise K/V are dense or packed rows (3-D maps).
// VAR: varlen or paged (per-sequence lengths from device arrays); only those
// instances carry the sorted schedule.
template <int D, bool PAGED, bool FP8, bool VAR>
__global__ void __launch_bounds__(kThreads, 1)
fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, __nv_bfloat16* __restrict__ o,
                float* __restrict__ lse, const int* __restrict__ cu_q,
                const int* __restrict__ cu_k, int B, int H, int Hkv, int n, int m, int total_q,
                int total_k, int num_pairs, float scale_log2, int causal, int lse_stride_h,
                int lse_stride_b, const int* __restrict__ block_table,
                const int* __restrict__ seq_lens, int max_blocks, int num_pages, float out_scale,
                int sched_sorted, int num_split, int* status) {
  using C = Cfg<D, FP8>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Shared sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int BH = B * H;
  const int* const seq_lens_p = PAGED ? seq_lens : nullptr;
  auto unit_bt = [&](int b, int h, int t) {
    return make_unit(b, h, t, H, Hkv, n, m, causal, cu_q, cu_k, total_q, total_k, seq_lens_p,
                     max_blocks);
  };
  // Dense: units are numbered heaviest first, pair index descending, then
  // (b, h).  Sorted (varlen and paged, few combinations): every CTA builds the
  // same list of (sequence, pair) combinations ordered by K/V tiles
  // descending (ties by index), and unit u is head u % H of entry u / H.
  if (VAR && sched_sorted) {
    const int C = B * num_pairs;
    if (threadIdx.x == 0) sh.n_order = 0;
    __syncthreads();
    for (int c = threadIdx.x; c < C; c += blockDim.x) {
      const Unit U = unit_bt(c / num_pairs, 0, c % num_pairs);
      if (U.bad) atomicExch(status, kDevInvalidArg);  // skipped, touches nothing
      // a unit with query rows but no keys still writes O = 0 and LSE = -inf;
      // the count saturates (a 16-bit wrap could reach 0 and drop the unit)
      sh.work[c] = (uint16_t)(U.rows ? min(1 + U.n_kv[0] + U.n_kv[1], 65535) : 0);
    }
    __syncthreads();
    int mine = 0;
    for (int c = threadIdx.x; c < C; c += blockDim.x) {
      const int w = sh.work[c];
      int rank = 0;
      for (int c2 = 0; c2 < C; ++c2) {
        const int w2 = sh.work[c2];
        rank += (w2 > w) || (w2 == w && c2 < c);
      }
      sh.order[rank] = (uint16_t)c;
      mine += w > 0;
    }
    if (mine) atomicAdd(&sh.n_order, mine);
    __syncthreads();
  }
  // Dense: the last num_split pair units (the partial last wave) are run as
  // 2 * num_split split units, one per query tile, so that wave finishes in
  // about half a unit's time.
  const int num_units = VAR && sched_sorted ? H * sh.n_order : BH * num_pairs + (VAR ? 0 : num_split);
  auto unit_at = [&](int u) {
    if (VAR && sched_sorted) {
      const int c = sh.order[u / H];
      return unit_bt(c / num_pairs, u % H, c % num_pairs);
    }
    const int base = BH * num_pairs - (VAR ? 0 : num_split);
    const int r = u < base ? u : base + (u - base) / 2;
    const int bh = r % BH;
    const Unit R = unit_bt(bh / H, bh % H, num_pairs - 1 - r / BH);
    return u < base ? R : split_unit(R, (u - base) & 1);
  };
#define FA_UNIT(u) unit_at(u)
  // k-th unit of this CTA: waves of gridDim.x units in snake order (even waves
  // left to right, odd waves right to left), which evens out the per-CTA sum
  // of the heaviest-first unit sizes
  auto unit_of = [&](int k) {
    const int g = (int)gridDim.x;
    return k * g + ((k & 1) ? g - 1 - (int)blockIdx.x : (int)blockIdx.x);
  };

  uint8_t* sQ = smem;                        // [2][kChunks][128 rows][128 B]
  uint8_t* sKV = smem + C::kQBytes;          // [kStages][kChunks (+1 of ones)][128 rows][128 B]

  const uint32_t bar_q = ptx::smem_u32(&sh.q_full[0]);
  const uint32_t bar_qe = ptx::smem_u32(&sh.q_empty[0]);
  const uint32_t bar_s = ptx::smem_u32(&sh.s_full[0]);
  const uint32_t bar_p = ptx::smem_u32(&sh.p_full[0]);
  const uint32_t bar_o = ptx::smem_u32(&sh.o_done[0]);
  const uint32_t bar_oe = ptx::smem_u32(&sh.o_empty[0]);
  const uint32_t bar_kvf = ptx::smem_u32(&sh.kv_full[0]);
  const uint32_t bar_kve = ptx::smem_u32(&sh.kv_empty[0]);
  const uint32_t bar_drain = ptx::smem_u32(&sh.drain);
  const uint32_t bar_fix = ptx::smem_u32(&sh.fix);
  const uint32_t bar_mf = ptx::smem_u32(&sh.merge_full);
  const uint32_t bar_me = ptx::smem_u32(&sh.merge_empty);
  volatile int* abort_flag = &sh.abort;

  if (threadIdx.x == 0) {
    #pragma unroll
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(bar_q + 8 * i, 1);
      ptx::mbar_init(bar_qe + 8 * i, 1);
      ptx::mbar_init(bar_s + 8 * i, 1);
      ptx::mbar_init(bar_p + 8 * i, kBlockM);
      ptx::mbar_init(bar_o + 8 * i, 1);
      ptx::mbar_init(bar_oe + 8 * i, kBlockM);
    }
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(bar_kvf + 8 * s, 1);
      ptx::mbar_init(bar_kve + 8 * s, 1);
    }
    ptx::mbar_init(bar_drain, 1);
    ptx::mbar_init(bar_fix, 1);
    ptx::mbar_init(bar_mf, kBlockM);
    ptx::mbar_init(bar_me, kBlockM);
    sh.abort = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if constexpr (C::kOnes) {
    // the block of ones behind every ring slot's tile: bf16 1.0 in every
    // element, so the swizzle does not matter; K and V loads never reach it
    constexpr int kWords = C::kTileBytes / 16;
    for (int idx = threadIdx.x; idx < C::kStages * kWords; idx += kThreads)
      *reinterpret_cast<uint4*>(sKV + (idx / kWords) * C::kSlotBytes + C::kTileBytes +
                                (idx % kWords) * 16) =
          make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    ptx::fence_proxy_async_smem();   // visible to the tensor core after the barrier below
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
      // ---------------------------------------------------------- producer
      // The whole warp walks the schedule; lane 0 issues the copies, and in
      // paged mode all lanes zero the V rows past a sequence's end.
      if (lane == 0) {
        ptx::prefetch_tmap(&tmQ);
        ptx::prefetch_tmap(&tmK);
        ptx::prefetch_tmap(&tmV);
      }
      // Q is read once; K and V are read again by the other query-tile pairs
      // of the head, so they are the ones L2 should keep
      const uint64_t pol_q = ptx::policy_evict_first();
      const uint64_t pol_kv = ptx::policy_evict_last();
      int li = 0;                 // K/V loads issued (K(j), V(j) alternate)
      int nq[2] = {0, 0};         // Q loads issued per tile
      int nfix = 0;               // V tiles zero-fixed (paged)
      bool fix_pending = false;
      bool ok = true;
      for (int k = 0; k * (int)gridDim.x < num_units && ok; ++k) {
        const int u = unit_of(k);
        if (u >= num_units) continue;
        const Unit U = FA_UNIT(u);
        if (U.bad && lane == 0) atomicExch(status, kDevInvalidArg);  // skip it, touch nothing
        if (!U.rows) continue;
        #pragma unroll
        for (int i = 0; i < 2 && ok; ++i) {
          if (U.n_kv[i] == 0) continue;
          // the previous unit's last S_i MMA must be done with Q_i
          if (!(ok = ptx::mbar_wait(bar_qe + 8 * i, (nq[i] & 1) ^ 1, status, abort_flag))) break;
          if (lane == 0) {
            const uint32_t dst = ptx::smem_u32(sQ + i * C::kTileBytes);
            ptx::mbar_arrive_expect_tx(bar_q + 8 * i, C::kTileBytes);
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c)
              ptx::tma_load_3d_hint(dst + c * 16384, &tmQ, C::kChunkElems * c, U.h,
                                    U.q_row0 + U.q_start[i], bar_q + 8 * i, pol_q);
          }
          ++nq[i];
        }
        // one K (which 0) or V (which 1) tile load into the next ring slot;
        // false if a wait failed
        auto issue_kv = [&](int which, int j) __attribute__((always_inline)) -> bool {
            const int slot = li % C::kStages;
            if (!ptx::mbar_wait(bar_kve + 8 * slot, ((li / C::kStages) & 1) ^ 1, status, abort_flag))
              return false;
            __syncwarp();
            uint8_t* tile = sKV + slot * C::kSlotBytes;
            const uint32_t dst = ptx::smem_u32(tile);
            const CUtensorMap* map = which == 0 ? &tmK : &tmV;
            const int rows_valid = min(kBlockN, U.kv_len - j * kBlockN);
            // A V tile whose rows past the sequence's end hold something else
            // (a cache page may hold anything; in a packed batch they are the
            // next sequence's rows) lands on the fix barrier first: those
            // keys' weights are exactly 0, but 0 * inf and 0 * NaN are NaN,
            // so the rows are zeroed before the MMA may read the tile.  Dense
            // tiles need no fix: their 4-D view reads zeros past a batch
            // element's last row, as the packed view does past the buffer.
            bool fix = false;
            if constexpr (PAGED) fix = which == 1 && rows_valid < kBlockN;
            else if constexpr (VAR)
              fix = which == 1 && rows_valid < kBlockN && U.k_row0 + U.kv_len < total_k;
            const uint32_t bar = fix ? bar_fix : bar_kvf + 8 * slot;
            if constexpr (PAGED) {
              const int npages = (rows_valid + 15) / 16;
              // lane 0 posts the byte count (the barrier's one arrival, so the
              // phase cannot complete before it), then lane pg looks up page
              // pg and issues its boxes: the page copies go out in parallel
              if (lane == 0) ptx::mbar_arrive_expect_tx(bar, npages * 16 * C::kRowBytes);
              __syncwarp();
              if (lane < npages) {
                const int pg = lane;
                int id = __ldg(block_table + (size_t)U.b * max_blocks + j * (kBlockN / 16) + pg);
                if (id < 0 || id >= num_pages) {
                  atomicExch(status, kDevBadBlockTable);
                  id = 0;
                }
                const int row = (id * Hkv + U.hk) * 16;
#pragma unroll
                for (int c = 0; c < C::kChunks; ++c)
                  ptx::tma_load_2d(dst + c * 16384 + pg * 2048, map, C::kChunkElems * c, row, bar);
              }
            } else {
              if (lane == 0) {
                ptx::mbar_arrive_expect_tx(bar, C::kTileBytes);
#pragma unroll
                for (int c = 0; c < C::kChunks; ++c) {
                  if constexpr (VAR)
                    ptx::tma_load_3d_hint(dst + c * 16384, map, C::kChunkElems * c, U.hk,
                                          U.k_row0 + j * kBlockN, bar, pol_kv);
                  else
                    ptx::tma_load_4d_hint(dst + c * 16384, map, C::kChunkElems * c, U.hk,
                                          j * kBlockN, U.b, bar, pol_kv);
                }
              }
            }
            if (fix) {
              fix_pending = true;
              if (!ptx::mbar_wait(bar_fix, nfix & 1, status, abort_flag)) return false;
              fix_pending = false;
              ++nfix;
              const int zero_rows = kBlockN - rows_valid;
              for (int idx = lane; idx < zero_rows * 8 * C::kChunks; idx += 32) {
                const int c = idx / (zero_rows * 8);
                const int rem = idx % (zero_rows * 8);
                const int row = rows_valid + rem / 8;
                *reinterpret_cast<uint4*>(tile + c * 16384 + row * 128 + (rem % 8) * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
              }
              ptx::fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) ptx::mbar_arrive(bar_kvf + 8 * slot);
            }
            ++li;
            return true;
        };
        const int n_kv_max = max(U.n_kv[0], U.n_kv[1]);
        if (!U.split) {
          for (int j = 0; j < n_kv_max && ok; ++j)
            for (int which = 0; which < 2 && ok; ++which) ok = issue_kv(which, j);  // K then V
        } else {
          // the MMA warp's order for a split unit: K_0(0), K_1(0), then per
          // step V_0(j), K_0(j+1), V_1(j), K_1(j+1) (tile i's K/V tiles
          // start at kv_first[i])
          #pragma unroll
          for (int i = 0; i < 2 && ok; ++i) ok = issue_kv(0, U.kv_first[i]);
          for (int j = 0; j < U.n_kv[0] && ok; ++j)
            #pragma unroll
            for (int i = 0; i < 2 && ok; ++i) {
              if (j < U.n_kv[i]) ok = issue_kv(1, U.kv_first[i] + j);
              if (ok && j + 1 < U.n_kv[i]) ok = issue_kv(0, U.kv_first[i] + j + 1);
            }
        }
      }
      if (!ok && lane == 0) {
        // let the last load of every slot, and of every Q tile, land before
        // shared memory is released
        for (int l = max(0, li - C::kStages); l < li; ++l)
          ptx::mbar_wait(bar_kvf + 8 * (l % C::kStages), (l / C::kStages) & 1, nullptr);
        #pragma unroll
        for (int i = 0; i < 2; ++i)
          if (nq[i] > 0) ptx::mbar_wait(bar_q + 8 * i, (nq[i] - 1) & 1, nullptr);
        if (fix_pending) ptx::mbar_wait(bar_fix, nfix & 1, nullptr);
      }
    } else if (warp == 1 && lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      const uint32_t q_addr[2] = {ptx::smem_u32(sQ), ptx::smem_u32(sQ + C::kTileBytes)};
      int lc = 0;                 // K/V loads consumed
      int nq[2] = {0, 0};         // Q tiles consumed
      int np[2] = {0, 0};         // P tiles consumed (= S tiles issued)
      int no[2] = {0, 0};         // units whose O_i was used
      bool ok = true;
      // Descriptors are built once; an MMA step only adds the byte offset of
      // its operand (in 16-byte units) to the start-address field (bits 0-13,
      // which cannot carry: shared addresses are below 256 KB).  This keeps
      // the single issuing thread to a few instructions per MMA.
      const uint64_t qdesc[2] = {ptx::smem_desc_sw128(q_addr[0], 16, 1024),
                                 ptx::smem_desc_sw128(q_addr[1], 16, 1024)};
      const uint64_t kdesc0 = ptx::smem_desc_sw128(ptx::smem_u32(sKV), 16, 1024);
      const uint64_t vdesc0 = ptx::smem_desc_sw128(ptx::smem_u32(sKV), 16384, 1024);
      auto issue_s = [&](int i, int slot) {
        const uint64_t kd = kdesc0 + (uint64_t)(slot * (C::kSlotBytes >> 4));
#pragma unroll
        for (int k = 0; k < C::kRowBytes / 32; ++k) {
          const uint32_t off = ((k >> 2) * 16384 + (k & 3) * 32) >> 4;
          if constexpr (FP8)
            ptx::mma_ss_f8(tbase + i * kBlockN, qdesc[i] + off, kd + off, C::kIdescS, k > 0);
          else
            ptx::mma_ss(tbase + i * kBlockN, qdesc[i] + off, kd + off, C::kIdescS, k > 0);
        }
      };
      // O_i += P_i V(j), issued once the softmax warps have stored all of
      // P_i; false if the wait failed
      auto issue_pv = [&](int i, int slot, int j) -> bool {
        const uint64_t vd = vdesc0 + (uint64_t)(slot * (C::kSlotBytes >> 4));
        if (!ptx::mbar_wait(bar_p + 8 * i, np[i] & 1, status, abort_flag)) return false;
        ptx::tc_fence_after();
#pragma unroll
        for (int k = 0; k < kBlockN / C::kKStep; ++k) {
          // a step covers kKStep keys: 8 packed P columns, kKStep V rows of 128 B
          const uint64_t bd = vd + (uint64_t)(k * C::kKStep * 8);
          if constexpr (FP8)
            ptx::mma_ts_f8(tbase + 256 + i * C::kOStride, tbase + i * kBlockN + k * 8, bd, C::kIdescO,
                           (j > 0 || k > 0) ? 1u : 0u);
          else
            ptx::mma_ts(tbase + 256 + i * C::kOStride, tbase + i * kBlockN + k * 8, bd, C::kIdescO,
                        (j > 0 || k > 0) ? 1u : 0u);
        }
        ++np[i];
        return true;
      };
      for (int k = 0; k * (int)gridDim.x < num_units && ok; ++k) {
        const int u = unit_of(k);
        if (u >= num_units) continue;
        const Unit U = FA_UNIT(u);
        if (!U.rows) continue;
        const int n_kv_max = max(U.n_kv[0], U.n_kv[1]);
        if (n_kv_max == 0) continue;
        #pragma unroll
        for (int i = 0; i < 2 && ok; ++i) {
          if (U.n_kv[i] == 0) continue;
          ok = ptx::mbar_wait(bar_q + 8 * i, nq[i] & 1, status, abort_flag);
          ++nq[i];
        }
        if (!ok) break;
        if (U.split) {
          // Split unit: each tile has its own K/V tiles, consumed in the
          // producer's order (K_0(0), K_1(0), then per step V_0(j), K_0(j+1),
          // V_1(j), K_1(j+1)); each slot is released right behind its MMAs.
          // wait for the next ring slot in load order; its index is lc - 1 after
          auto next_slot = [&]() -> bool {
            const bool w = ptx::mbar_wait(bar_kvf + 8 * (lc % C::kStages), (lc / C::kStages) & 1,
                                          status, abort_flag);
            ++lc;
            if (w) ptx::tc_fence_after();
            return w;
          };
          #pragma unroll
          for (int i = 0; i < 2 && ok; ++i) {
            if (!(ok = next_slot())) break;
            const int slot = (lc - 1) % C::kStages;
            issue_s(i, slot);
            ptx::tc_commit(bar_s + 8 * i);
            if (U.n_kv[i] == 1) ptx::tc_commit(bar_qe + 8 * i);
            ptx::tc_commit(bar_kve + 8 * slot);
          }
          for (int j = 0; j < U.n_kv[0] && ok; ++j) {
            #pragma unroll
            for (int i = 0; i < 2 && ok; ++i) {
              if (j >= U.n_kv[i]) continue;
              if (!(ok = next_slot())) break;
              const int slot = (lc - 1) % C::kStages;
              // K_i(j+1) before P_i(j), as in the pair loop below
              const bool nxt = j + 1 < U.n_kv[i];
              if (nxt && !(ok = next_slot())) break;
              const int sk = (lc - 1) % C::kStages;
              if (j == 0 && !(ok = ptx::mbar_wait(bar_oe + 8 * i, (no[i] & 1) ^ 1, status, abort_flag))) break;
              if (!(ok = issue_pv(i, slot, j))) break;
              if (j == U.n_kv[i] - 1) ptx::tc_commit(bar_o + 8 * i);
              ptx::tc_commit(bar_kve + 8 * slot);
              if (nxt) {
                issue_s(i, sk);
                ptx::tc_commit(bar_s + 8 * i);
                if (j + 2 == U.n_kv[i]) ptx::tc_commit(bar_qe + 8 * i);
                ptx::tc_commit(bar_kve + 8 * sk);
              }
            }
          }
          #pragma unroll
          for (int i = 0; i < 2; ++i)
            if (U.n_kv[i] > 0) ++no[i];
          continue;
        }
        // prologue: S_i(0)
        {
          const int slot = lc % C::kStages;
          if (!(ok = ptx::mbar_wait(bar_kvf + 8 * slot, (lc / C::kStages) & 1, status, abort_flag))) break;
          ptx::tc_fence_after();
          #pragma unroll
          for (int i = 0; i < 2; ++i) {
            if (U.n_kv[i] == 0) continue;
            issue_s(i, slot);
            ptx::tc_commit(bar_s + 8 * i);
            if (U.n_kv[i] == 1) ptx::tc_commit(bar_qe + 8 * i);
          }
          ptx::tc_commit(bar_kve + 8 * slot);  // K(0)
        }
        for (int j = 0; j < n_kv_max && ok; ++j) {
          const int lv = lc + 2 * j + 1, sv = lv % C::kStages;
          const int lk = lc + 2 * j + 2, sk = lk % C::kStages;
          const bool has_next = j + 1 < n_kv_max;
          if (!(ok = ptx::mbar_wait(bar_kvf + 8 * sv, (lv / C::kStages) & 1, status, abort_flag))) break;
          // K(j+1) is waited for here, before P_0(j): it has landed long
          // before P_0(j) is ready, and a wait between P_0 V(j) and
          // S_0(j+1) would leave the tensor pipe idle behind P_0 V(j)
          if (has_next &&
              !(ok = ptx::mbar_wait(bar_kvf + 8 * sk, (lk / C::kStages) & 1, status, abort_flag)))
            break;
          ptx::tc_fence_after();
          // before the first P V of a unit, the previous unit's epilogue must
          // have read O_i out of tensor memory
          if (j < U.n_kv[0]) {
            if (j == 0 && !(ok = ptx::mbar_wait(bar_oe, (no[0] & 1) ^ 1, status, abort_flag))) break;
            if (!(ok = issue_pv(0, sv, j))) break;
            if (j == U.n_kv[0] - 1) ptx::tc_commit(bar_o);
          }
          // release K(j) (last read by S_i(j), issued in the previous
          // iteration) here, behind a burst of queued MMAs rather than in the
          // gap after S_1(j); K(0) was released in the prologue
          if (j > 0) ptx::tc_commit(bar_kve + 8 * ((lc + 2 * j) % C::kStages));
          if (j + 1 < U.n_kv[0]) {
            issue_s(0, sk);
            ptx::tc_commit(bar_s);
            if (j + 2 == U.n_kv[0]) ptx::tc_commit(bar_qe);
          }
          if (j < U.n_kv[1]) {
            if (j == 0 && !(ok = ptx::mbar_wait(bar_oe + 8, (no[1] & 1) ^ 1, status, abort_flag))) break;
            if (!(ok = issue_pv(1, sv, j))) break;
            if (j == U.n_kv[1] - 1) ptx::tc_commit(bar_o + 8);
          }
          ptx::tc_commit(bar_kve + 8 * sv);  // V(j)
          if (j + 1 < U.n_kv[1]) {
            issue_s(1, sk);
            ptx::tc_commit(bar_s + 8);
            if (j + 2 == U.n_kv[1]) ptx::tc_commit(bar_qe + 8);
          }
        }
        lc += 2 * n_kv_max;
        #pragma unroll
        for (int i = 0; i < 2; ++i)
          if (U.n_kv[i] > 0) ++no[i];
      }
      // no tcgen05.mma may still run when the tensor memory is released
      ptx::tc_commit(bar_drain);
      ptx::mbar_wait(bar_drain, 0, nullptr);
    }
  } else {
    ptx::setmaxnreg_inc<kSoftmaxRegs>();
    // ------------------------------------------------------------ softmax
    const int i = (warp - 4) / 4;             // query tile of this warpgroup
    const int quarter = warp & 3;             // tensor-memory lane quarter
    const int r = quarter * 32 + lane;        // row in the tile
    const uint32_t lane_base = tbase + ((uint32_t)(quarter * 32) << 16);
    const uint32_t s_col = lane_base + i * kBlockN;
    const uint32_t o_col = lane_base + 256 + i * C::kOStride;
    int ns = 0;    // S tiles consumed
    int nod[2] = {0, 0};   // units whose tile 0 / tile 1 had K/V tiles (o_done phases)
    int nsplit = 0;        // split units seen (merge barrier phases)
    bool ok = true;
    // 64 bytes of a row of O: rows are 2D bytes, so when O starts on a
    // 32-byte boundary every 32 bytes go out in one store (a whole sector),
    // half the store instructions and L2 writes of the 16-byte form
    const bool o32 = (reinterpret_cast<uintptr_t>(o) & 31u) == 0;
    auto store_o64 = [&](uint4* dst, const uint4 (&v)[4]) __attribute__((always_inline)) {
      if (o32) {
        ptx::st_global_v8(dst, v[0], v[1]);
        ptx::st_global_v8(dst + 2, v[2], v[3]);
      } else {
#pragma unroll
        for (int w = 0; w < 4; ++w) dst[w] = v[w];
      }
    };
    for (int k = 0; k * (int)gridDim.x < num_units && ok; ++k) {
      const int u = unit_of(k);
      if (u >= num_units) continue;
      const Unit U = FA_UNIT(u);
      if (!U.rows) continue;
      // (selects, not U.x[i]: a runtime index would put the unit in local memory)
      const int q_start = i == 0 ? U.q_start[0] : U.q_start[1];
      const int kv_first = i == 0 ? U.kv_first[0] : U.kv_first[1];
      const int qi = q_start + r;               // query index in the sequence
      const int nkv = i == 0 ? U.n_kv[0] : U.n_kv[1];
      float m_ref = -INFINITY;   // running reference (log2 units)
      bool max_first = false;    // this warp forms P max-first for the rest of the unit
      float l_run = 0.f;         // sum of the unrounded p: the LSE's l
      float l_p = 0.f;           // bf16: sum of the rounded p the P V MMA used (O's divisor)
      for (int j = 0; j < nkv; ++j) {
        // warp-uniform outcome: the tcgen05.ld/st below are warp-collective
        ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar_s + 8 * i, ns & 1, status, abort_flag));
        if (!ok) break;
        ++ns;
        ptx::tc_fence_after();
        // mask keys past the end and, causal, keys j > qi + (m - n): only tiles
        // that reach past the end or past the tile's first row's diagonal
        const int k0 = (kv_first + j) * kBlockN;
        const int diag = q_start + (U.kv_len - U.q_len);   // last key row q_start sees
        const bool masked = k0 + kBlockN > U.kv_len || (causal && k0 + kBlockN - 1 > diag);
        int vis = U.kv_len - k0;
        if (causal) vis = min(vis, qi + (U.kv_len - U.q_len) - k0 + 1);
        uint32_t sr[4][32];
        // S into registers.  Where the row max is wanted (a unit's first tile,
        // a max-first warp, the reload after a miss) and no key is masked, the
        // loads reduce it themselves (tcgen05.ld.red ... .max): the hardware
        // max of each thread's 32 columns, so the 43 three-input max of
        // row_max are not spent.  Masked tiles take row_max after masking,
        // since the loads would see the masked scores too.
        float mred = -INFINITY;
        bool have_mred = false;
        auto load_s = [&](bool want_max) {
          if (!masked && want_max) {
            float mc[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) ptx::tmem_ld32_max(s_col + c * 32, sr[c], mc[c]);
            ptx::tmem_wait_ld();
            mred = fmaxf(fmaxf(mc[0], mc[1]), fmaxf(mc[2], mc[3]));
            have_mred = true;
            return;
          }
#pragma unroll
          for (int c = 0; c < 4; ++c) ptx::tmem_ld32(s_col + c * 32, sr[c]);
          ptx::tmem_wait_ld();
          if (masked) {
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (c * 32 + e >= vis) sr[c][e] = __float_as_uint(-INFINITY);
          }
        };
        load_s(j == 0 || max_first);
        // From the second tile on, P is first formed against the current
        // reference without the row max.  Every p is at most the tile's row
        // sum, so a sum of at most 2^threshold shows that no score passed the
        // reference by more than the threshold: no raise is due, and this P
        // is exactly the one the max-first path forms.  Only a warp with a
        // larger sum (or a row with no reference yet) takes the max and forms
        // P again.  After such a miss the warp goes max-first for the rest of
        // the unit: misses come in runs (scores that keep climbing, as in rows
        // with a few dominant keys), and each costs a second pass.  Measured
        // on the hot ragged workload (d=128): 715 TFLOP/s retrying every tile,
        // 786 going max-first for 4 tiles, 821 for the rest of the unit.
        // (bf16: the first attempt stores nothing, so on a miss S is still
        // whole in tensor memory and is loaded again instead of being kept in
        // registers beside the packed P.)
        const uint64_t sc2 = ptx::f2_bits(scale_log2, scale_log2);
        float lsum = 0.f;
        bool full = true;
        uint32_t pp[64];   // bf16: this tile's packed P
        if (j > 0 && !max_first) {
          const float ref = m_ref == -INFINITY ? 0.f : m_ref;
          if constexpr (FP8) lsum = exp_pass<true>(sr, s_col, sc2, ptx::f2_bits(-ref, -ref));
          else lsum = exp_pack_bf16<false>(sr, s_col, sc2, ptx::f2_bits(-ref, -ref), pp);
          full = __any_sync(0xffffffffu, !(lsum <= kRaiseSum) || m_ref == -INFINITY);
          max_first = full;
          if constexpr (!FP8) {
            if (full) load_s(true);
            else ptx::tmem_st64(s_col, pp);
          }
        }
        if (full) {
          const float m_tile = (have_mred ? mred : row_max(sr)) * scale_log2;   // scale > 0: max commutes with it
          const bool raise =
              m_tile > m_ref + kRescaleThreshold || (m_ref == -INFINITY && m_tile > -INFINITY);
          float alpha = 1.f;
          if (raise) {
            alpha = m_ref == -INFINITY ? 1.f : ptx::ex2(m_ref - m_tile);
            m_ref = m_tile;
            l_run *= alpha;
            l_p *= alpha;
          }
          const float ref = m_ref == -INFINITY ? 0.f : m_ref;
          // rescale acc when this warp raised a reference after the first
          // tile: no P V of this tile may run before it
          if (__any_sync(0xffffffffu, raise && j > 0 && alpha != 1.f)) {
#pragma unroll 1
            for (int c = 0; c < (C::kON + 31) / 32; ++c) {   // with l_p's columns
              uint32_t ov[32];
              ptx::tmem_ld32(o_col + c * 32, ov);
              ptx::tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
              ptx::tmem_st32(o_col + c * 32, ov);
            }
          }
          if constexpr (FP8) lsum = exp_pass<true>(sr, s_col, sc2, ptx::f2_bits(-ref, -ref));
          else lsum = exp_pack_bf16<true>(sr, s_col, sc2, ptx::f2_bits(-ref, -ref), pp);
        }
        // all of P_i sits in tensor memory: hand it to the MMA warp
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar_p + 8 * i);
        l_run += lsum;
        // O is divided by the sum of the p the MMA multiplied (rounded to
        // bf16), not by the exact sum: then a row that one key dominates gets
        // that key's V row back to within fp32 rounding, where the exact sum
        // would leave the rounding of that key's p (up to 2^-8 relative) in O.
        // Done after the hand-off, while the MMAs run.
        if constexpr (!FP8 && !C::kOnes) l_p += sum_packed_bf16(pp);
      }
      if (!ok) break;

      // ---- epilogue: O = acc / l (bf16), LSE = (ref + log2 l) ln 2
      const bool row_valid = qi < U.q_len;
      const size_t orow = (size_t)(U.q_row0 + qi) * H + U.h;
      const int ph_o0 = nod[0] & 1, ph_o1 = nod[1] & 1, ph_m = nsplit & 1;
      if (U.n_kv[0] > 0) ++nod[0];
      if (U.n_kv[1] > 0) ++nod[1];
      if (U.split) {
        ++nsplit;
        if (i == 1) {
          // hand this row's state to warpgroup 0, which merges the two halves
          ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar_me, ph_m ^ 1, status, abort_flag));
          if (!ok) break;
          sh.mstat[r][0] = m_ref;
          sh.mstat[r][1] = l_run;
          sh.mstat[r][2] = l_p;
          ptx::mbar_arrive(bar_mf);
          continue;
        }
        // M = max of the two references, a_i = 2^(m_i - M) (0 for a state
        // that saw no key); O = (a_0 acc_0 + a_1 acc_1) / (a_0 l_0 + a_1 l_1)
        // with the rounded sums, LSE from the exact ones
        ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar_o, ph_o0, status, abort_flag) &&
                                         ptx::mbar_wait(bar_o + 8, ph_o1, status, abort_flag) &&
                                         ptx::mbar_wait(bar_mf, ph_m, status, abort_flag));
        if (!ok) break;
        ptx::tc_fence_after();
        const uint32_t o_col1 = lane_base + 256 + C::kOStride;   // O_1: the other key range
        const float m1 = sh.mstat[r][0], l1 = sh.mstat[r][1];
        float lp1 = sh.mstat[r][2];
        if constexpr (C::kOnes) {   // both rounded sums sit in column D of their O
          uint32_t t0[32], t1[32];
          ptx::tmem_ld32(o_col + D, t0);
          ptx::tmem_ld32(o_col1 + D, t1);
          ptx::tmem_wait_ld();
          l_p = __uint_as_float(t0[0]);
          lp1 = __uint_as_float(t1[0]);
        }
        ptx::mbar_arrive(bar_me);
        const float M = fmaxf(m_ref, m1);
        const float a0 = m_ref == -INFINITY ? 0.f : ptx::ex2(m_ref - M);
        const float a1 = m1 == -INFINITY ? 0.f : ptx::ex2(m1 - M);
        const float l_all = a0 * l_run + a1 * l1;
        const float lo_all = FP8 ? l_all : a0 * l_p + a1 * lp1;
        const float inv = lo_all > 0.f ? out_scale / lo_all : 0.f;
        const float c0 = a0 * inv, c1 = a1 * inv;
        const bool store = row_valid && FA_IN_BOUNDS(orow, (size_t)total_q * H, status);
        uint4* dst = reinterpret_cast<uint4*>(o + orow * D);
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t x0[32], x1[32];
          ptx::tmem_ld32(o_col + c * 32, x0);
          ptx::tmem_ld32(o_col1 + c * 32, x1);
          ptx::tmem_wait_ld();
          if (store) {
            uint4 v[4];
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              float f[8];
#pragma unroll
              for (int e = 0; e < 8; ++e)
                f[e] = __uint_as_float(x0[8 * w + e]) * c0 + __uint_as_float(x1[8 * w + e]) * c1;
              v[w].x = ptx::pack_bf16x2(f[0], f[1]);
              v[w].y = ptx::pack_bf16x2(f[2], f[3]);
              v[w].z = ptx::pack_bf16x2(f[4], f[5]);
              v[w].w = ptx::pack_bf16x2(f[6], f[7]);
            }
            store_o64(dst + c * 4, v);
          }
        }
        // both O accumulators may now be overwritten by the next unit
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar_oe);
        ptx::mbar_arrive(bar_oe + 8);
        if (store) {
          const size_t li = (size_t)U.b * lse_stride_b + (size_t)U.h * lse_stride_h +
                            (U.q_row0 - (cu_q ? 0 : U.b * n)) + qi;
          if (lse != nullptr && FA_IN_BOUNDS(li, (size_t)total_q * H, status))
            lse[li] = l_all > 0.f ? (M + __log2f(l_all)) * kLn2 : -INFINITY;
        }
        continue;
      }
      uint32_t ov[D / 32][32];
      if (nkv > 0) {
        ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar_o + 8 * i, i == 0 ? ph_o0 : ph_o1, status,
                                                    abort_flag));
        if (!ok) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) ptx::tmem_ld32(o_col + c * 32, ov[c]);
        if constexpr (C::kOnes) {   // the rounded sum from O's column D
          uint32_t t[32];
          ptx::tmem_ld32(o_col + D, t);
          ptx::tmem_wait_ld();
          l_p = __uint_as_float(t[0]);
        }
        ptx::tmem_wait_ld();
        // O_i may now be overwritten by the next unit's first P V
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar_oe + 8 * i);
      } else {
#pragma unroll
        for (int c = 0; c < D / 32; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[c][e] = 0u;
      }
      // O has total_q * H rows of D (dense: total_q = B * n); LSE as many entries
      if (row_valid && FA_IN_BOUNDS(orow, (size_t)total_q * H, status)) {
        // O's divisor (bf16: the rounded sum, positive exactly when l_run is:
        // a normal fp32 p rounds to a normal bf16) and the LSE's l
        const float l_o = FP8 ? l_run : l_p;
        const float inv = l_o > 0.f ? out_scale / l_o : 0.f;
        uint4* dst = reinterpret_cast<uint4*>(o + orow * D);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint4 v[4];
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            v[w].x = ptx::pack_bf16x2(__uint_as_float(ov[c][8 * w + 0]) * inv, __uint_as_float(ov[c][8 * w + 1]) * inv);
            v[w].y = ptx::pack_bf16x2(__uint_as_float(ov[c][8 * w + 2]) * inv, __uint_as_float(ov[c][8 * w + 3]) * inv);
            v[w].z = ptx::pack_bf16x2(__uint_as_float(ov[c][8 * w + 4]) * inv, __uint_as_float(ov[c][8 * w + 5]) * inv);
            v[w].w = ptx::pack_bf16x2(__uint_as_float(ov[c][8 * w + 6]) * inv, __uint_as_float(ov[c][8 * w + 7]) * inv);
          }
          store_o64(dst + c * 4, v);
        }
        const size_t li = (size_t)U.b * lse_stride_b + (size_t)U.h * lse_stride_h +
                          (U.q_row0 - (cu_q ? 0 : U.b * n)) + qi;
        if (lse != nullptr && FA_IN_BOUNDS(li, (size_t)total_q * H, status))
          lse[li] = l_run > 0.f ? (m_ref + __log2f(l_run)) * kLn2 : -INFINITY;
      }
    }
  }
#undef FA_UNIT

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tbase, 512);
  }
}

template <int D, bool PAGED, bool FP8>
cudaError_t launch(const FwdParams& p, cudaStream_t stream, const char** why) {
  using C = Cfg<D, FP8>;
  const CUtensorMapDataType dt = FP8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const bool varlen = p.cu_q != nullptr;
  // 3-D views (dim, head, token row) of Q, K, V; out-of-range rows read as 0.
  const uint64_t q_rows = varlen ? (uint64_t)(p.total_q > 0 ? p.total_q : 1) : (uint64_t)p.B * p.n;
  const uint64_t k_rows = varlen ? (uint64_t)(p.total_k > 0 ? p.total_k : 1) : (uint64_t)p.B * p.m;
  CUtensorMap tq, tk, tv;
  const uint32_t box[3] = {(uint32_t)C::kChunkElems, 1, 128};
  {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)p.H, q_rows};
    const uint64_t strides[2] = {(uint64_t)C::kRowBytes, (uint64_t)p.H * C::kRowBytes};
    if (!make_tmap_bf16(&tq, p.q, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, dt)) {
      *why = "tensor map for q";
      return cudaErrorInvalidValue;
    }
  }
  if (PAGED) {
    // 2-D views (dim, page row) of the caches; one box = one page of one kv head
    const uint64_t dims[2] = {(uint64_t)D, (uint64_t)p.num_pages * p.Hkv * 16};
    const uint64_t strides[1] = {(uint64_t)C::kRowBytes};
    const uint32_t pbox[2] = {(uint32_t)C::kChunkElems, 16};
    if (!make_tmap_bf16(&tk, p.k, 2, dims, strides, pbox, CU_TENSOR_MAP_SWIZZLE_128B, dt) ||
        !make_tmap_bf16(&tv, p.v, 2, dims, strides, pbox, CU_TENSOR_MAP_SWIZZLE_128B, dt)) {
      *why = "tensor map for the k/v caches";
      return cudaErrorInvalidValue;
    }
  } else if (varlen) {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)p.Hkv, k_rows > 0 ? k_rows : 1};
    const uint64_t strides[2] = {(uint64_t)C::kRowBytes, (uint64_t)p.Hkv * C::kRowBytes};
    if (!make_tmap_bf16(&tk, p.m > 0 ? p.k : p.q, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, dt) ||
        !make_tmap_bf16(&tv, p.m > 0 ? p.v : p.q, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, dt)) {
      *why = "tensor map for k/v";
      return cudaErrorInvalidValue;
    }
  } else {
    // 4-D views (dim, head, token row, batch element) of dense K and V: a
    // tile past an element's last row reads zeros, never the next element
    const uint64_t m_rows = p.m > 0 ? (uint64_t)p.m : 1;
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)p.Hkv, m_rows, (uint64_t)p.B};
    const uint64_t strides[3] = {(uint64_t)C::kRowBytes, (uint64_t)p.Hkv * C::kRowBytes,
                                 m_rows * p.Hkv * C::kRowBytes};
    const uint32_t box4[4] = {(uint32_t)C::kChunkElems, 1, 128, 1};
    if (!make_tmap_bf16(&tk, p.m > 0 ? p.k : p.q, 4, dims, strides, box4, CU_TENSOR_MAP_SWIZZLE_128B, dt) ||
        !make_tmap_bf16(&tv, p.m > 0 ? p.v : p.q, 4, dims, strides, box4, CU_TENSOR_MAP_SWIZZLE_128B, dt)) {
      *why = "tensor map for k/v";
      return cudaErrorInvalidValue;
    }
  }
  const int num_pairs = (p.n + 2 * kBlockM - 1) / (2 * kBlockM);
  const long long units = (long long)p.B * p.H * num_pairs;
  int sms = 0;
  {
    int dev = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) {
      *why = "query SM count";
      return e;
    }
  }
  // Persistent, one CTA per SM (the shared-memory footprint admits one),
  // units in snake order: dense, and varlen or paged with few (sequence,
  // pair) combinations (the kernel sorts them by size).  Otherwise one CTA
  // per unit, so the hardware block scheduler balances units whose sizes
  // depend on lengths the host does not know (idle units exit at once).
  const bool sorted = varlen && (long long)p.B * num_pairs <= kMaxSortedCombos;
  const int grid = varlen && !sorted ? (int)units : (int)(units < sms ? units : sms);
  // Dense and non-causal (units of equal size): when the last wave of pair
  // units would leave at least half the CTAs idle, those units run as twice
  // as many split units of about half the length.  Causal units already
  // shrink towards the end of the heaviest-first order.
  int num_split = 0;
  if (!varlen && !PAGED && !p.causal && (p.m + kBlockN - 1) / kBlockN >= 2) {
    const long long tail = units % grid;
    if (tail > 0 && 2 * tail <= grid) num_split = (int)tail;
  }
  // LSE layout: dense [B][H][n] ; varlen and paged [H][Tq]
  const int lse_stride_h = varlen ? p.total_q : p.n;
  const int lse_stride_b = varlen ? 0 : p.H * p.n;
  // e4m3 operands hold x / descale: the q and k descales fold into the score
  // scale, the v descale into the epilogue's 1 / l
  const float scale_log2 = p.scale * kLog2e * (FP8 ? p.q_descale * p.k_descale : 1.f);
  const float out_scale = FP8 ? p.v_descale : 1.f;
  auto go = [&](auto kernel) -> cudaError_t {
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (err != cudaSuccess) {
      *why = "cudaFuncSetAttribute(fwd_bf16)";
      return err;
    }
    kernel<<<grid, kThreads, C::kSmem, stream>>>(
        tq, tk, tv, static_cast<__nv_bfloat16*>(p.o), p.lse, p.cu_q, p.cu_k, p.B, p.H, p.Hkv, p.n,
        p.m, varlen ? p.total_q : p.B * p.n, varlen ? p.total_k : p.B * p.m, num_pairs, scale_log2,
        p.causal, lse_stride_h, lse_stride_b, p.block_table, p.seq_lens, p.max_blocks, p.num_pages,
        out_scale, sorted ? 1 : 0, num_split, p.status);
    err = cudaGetLastError();
    if (err != cudaSuccess) *why = "fwd_bf16 launch";
    return err;
  };
  if constexpr (PAGED) {
    return go(fwd_bf16_kernel<D, true, FP8, true>);
  } else if constexpr (FP8) {   // the C ABI's e4m3 entry is dense only
    if (varlen) {
      *why = "fwd e4m3: dense only";
      return cudaErrorInvalidValue;
    }
    return go(fwd_bf16_kernel<D, false, true, false>);
  } else {
    return varlen ? go(fwd_bf16_kernel<D, false, false, true>) : go(fwd_bf16_kernel<D, false, false, false>);
  }
}

}  // namespace

cudaError_t launch_fwd_bf16(const FwdParams& p, cudaStream_t stream, const char** why) {
  const bool paged = p.block_table != nullptr;
  if (p.fp8) {
    if (p.d == 128 && p.dv == 128 && !paged) return launch<128, false, true>(p, stream, why);
    *why = "fwd e4m3: supported d == dv == 128, dense";
    return cudaErrorInvalidValue;
  }
  if (p.d == 128 && p.dv == 128)
    return paged ? launch<128, true, false>(p, stream, why) : launch<128, false, false>(p, stream, why);
  if (p.d == 64 && p.dv == 64)
    return paged ? launch<64, true, false>(p, stream, why) : launch<64, false, false>(p, stream, why);
  *why = "fwd_bf16: unsupported head dim";
  return cudaErrorInvalidValue;
}

}  // namespace fa
