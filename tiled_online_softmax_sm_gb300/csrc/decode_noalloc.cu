// fa_paged_decode_noalloc: the paged split-KV decode without a caller
// workspace and without any allocation.
//
// Who needs it: code that cannot call cudaMalloc on its own.  A plugin living
// inside a host framework must take all device memory from that framework's
// allocator, and a serving loop that has finished start-up must not allocate
// (cudaMalloc can synchronise the whole device and stall every stream).  Such
// callers still own the inputs and outputs; the split partials, which the
// ordinary entry point places in a caller-provided workspace, live here in one
// fixed array of device memory that the library declares itself.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds it (kNoAllocScratchBytes) until the process exits.  Host code
// cannot pass the variable's name to a kernel (on the host it only stands in
// for the symbol); its device address is looked up by cudaGetSymbolAddress,
// with the device current, on the first call made on that device, and kept.
// The address belongs to the CUDA context the module is loaded in, so it is
// kept per context id: after a cudaDeviceReset (a new context, where the array
// has a new address) the next call looks it up again instead of handing the
// kernels a stale pointer.
//
// All calls share the array and it keeps the previous call's contents.  When
// a call completes with the device status clear, the partials kernel has
// overwritten every (m, l, o) triple the merge reads, so nothing has to be
// cleared first.  After FA_ERR_TIMEOUT some warps returned without writing
// their triples and the merge read the previous call's: O and LSE of that
// call are undefined.  Two calls whose work overlaps on the GPU (other
// streams, other host threads) race on the array and corrupt each other's
// results: serialise them.
#include <cuda_runtime.h>
#include <math.h>
#include <mutex>
#include <stdint.h>
#include <stdio.h>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace fa {
fa_status api_fail(fa_status st, const char* msg);
fa_status api_status_ptr(int** out);
}  // namespace fa

namespace {

constexpr size_t kNoAllocScratchBytes = FA_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxContexts = 64;
struct ScratchAddr {
  unsigned long long ctx;
  void* ptr;
};
ScratchAddr g_scratch_addr[kMaxContexts] = {};
int g_scratch_next = 0;
std::mutex g_scratch_mutex;

// Device address of the scratch array in the context current on this thread
// (the current device's primary context unless the caller bound another).
fa_status scratch_address(void** out) {
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  unsigned long long ctx = 0;
  if (fa::current_context_id(&ctx)) {
    for (const ScratchAddr& a : g_scratch_addr)
      if (a.ptr != nullptr && a.ctx == ctx) {
        *out = a.ptr;
        return FA_OK;
      }
  }
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || p == nullptr) {
    char msg[256];
    snprintf(msg, sizeof(msg), "fa_paged_decode_noalloc: cudaGetSymbolAddress(scratch): %s",
             cudaGetErrorString(e));
    return fa::api_fail(FA_ERR_CUDA, msg);
  }
  if (fa::current_context_id(&ctx)) {   // else (no context ids) look it up every call
    g_scratch_addr[g_scratch_next] = ScratchAddr{ctx, p};
    g_scratch_next = (g_scratch_next + 1) % kMaxContexts;
  }
  *out = p;
  return FA_OK;
}

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

extern "C" fa_status fa_paged_decode_noalloc(const void* q, const void* k_cache,
                                             const void* v_cache, const int* block_table,
                                             const int* seq_lens, void* o, float* lse,
                                             int num_seqs, int H, int Hkv, int d, int dv,
                                             int page_size, int num_pages, int max_blocks_per_seq,
                                             int num_splits, float scale, void* stream) {
  char msg[256];
  if (num_seqs < 0 || num_pages < 0 || max_blocks_per_seq < 0)
    return fa::api_fail(FA_ERR_INVALID_ARG, "fa_paged_decode_noalloc: negative size");
  if (H <= 0 || Hkv <= 0 || H % Hkv != 0)
    return fa::api_fail(FA_ERR_INVALID_ARG, "fa_paged_decode_noalloc: need H > 0, Hkv > 0, H % Hkv == 0");
  if (num_splits < 1 || num_splits > 64)
    return fa::api_fail(FA_ERR_INVALID_ARG, "fa_paged_decode_noalloc: num_splits outside [1, 64]");
  if (!(scale > 0.f) || scale == INFINITY)
    return fa::api_fail(FA_ERR_INVALID_ARG, "fa_paged_decode_noalloc: scale must be positive and finite");
  if (d != 128 || dv != 128 || page_size != 16 || H / Hkv > 16)
    return fa::api_fail(FA_ERR_UNSUPPORTED,
                        "fa_paged_decode_noalloc: supported d == dv == 128, page_size 16, H/Hkv <= 16");
  const size_t need = fa_paged_decode_workspace_size(num_seqs, H, dv, num_splits);
  if (need > kNoAllocScratchBytes) {
    snprintf(msg, sizeof(msg),
             "fa_paged_decode_noalloc: the split partials need %zu bytes, more than the fixed "
             "scratch of %zu bytes (use fewer sequences or splits, or fa_paged_decode)",
             need, kNoAllocScratchBytes);
    return fa::api_fail(FA_ERR_WORKSPACE, msg);
  }
  if (num_seqs == 0) return FA_OK;
  if (q == nullptr || o == nullptr || block_table == nullptr || seq_lens == nullptr ||
      k_cache == nullptr || v_cache == nullptr)
    return fa::api_fail(FA_ERR_INVALID_ARG, "fa_paged_decode_noalloc: null pointer");
  if (num_pages == 0 || max_blocks_per_seq == 0)
    return fa::api_fail(FA_ERR_INVALID_ARG, "fa_paged_decode_noalloc: empty page pool or block table");
  // page rows (page * Hkv + head) * 16 are 32-bit in the kernels (the units,
  // sequences x heads x splits, are bounded by the scratch size above)
  if ((long long)num_pages * Hkv * 16 > 0x7fffffffLL)
    return fa::api_fail(FA_ERR_UNSUPPORTED, "fa_paged_decode_noalloc: page pool too large");
  const uintptr_t mis = (reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
                         reinterpret_cast<uintptr_t>(v_cache) | reinterpret_cast<uintptr_t>(o)) & 15u;
  if (mis || (reinterpret_cast<uintptr_t>(lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return fa::api_fail(FA_ERR_INVALID_ARG, "fa_paged_decode_noalloc: misaligned pointer");

  int* status = nullptr;
  fa_status st = fa::api_status_ptr(&status);
  if (st != FA_OK) return st;
  void* scratch = nullptr;
  if ((st = scratch_address(&scratch)) != FA_OK) return st;

  // the partials carved as in fa_paged_decode's workspace (no ticket words:
  // the merge runs as its own launch)
  const size_t tri = (size_t)num_seqs * H * num_splits;
  char* ws = static_cast<char*>(scratch);
  float* part_m = reinterpret_cast<float*>(ws);
  float* part_l = reinterpret_cast<float*>(ws + round256(tri * sizeof(float)));
  float* part_o = reinterpret_cast<float*>(ws + 2 * round256(tri * sizeof(float)));
  fa::DecodeParams p{q, k_cache, v_cache, block_table, seq_lens, num_seqs, H, Hkv, d, dv,
                     page_size, num_pages, max_blocks_per_seq, num_splits, scale,
                     part_m, part_l, part_o, status};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = fa::launch_decode_partials(p, s);
  if (e != cudaSuccess) {
    snprintf(msg, sizeof(msg), "fa_paged_decode_noalloc partials launch: %s", cudaGetErrorString(e));
    return fa::api_fail(FA_ERR_CUDA, msg);
  }
  fa::CombineParams c{part_m, part_l, part_o, o, lse, num_seqs, H, num_splits, dv};
  e = fa::launch_split_combine(c, s);
  if (e != cudaSuccess) {
    snprintf(msg, sizeof(msg), "fa_paged_decode_noalloc merge launch: %s", cudaGetErrorString(e));
    return fa::api_fail(FA_ERR_CUDA, msg);
  }
  return FA_OK;
}
