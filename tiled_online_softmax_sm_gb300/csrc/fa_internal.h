// Internal launch interface between the C ABI layer (api.cu) and the kernel
// translation units.  Host-side only; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace fa {

// Id of the CUDA context current on the calling thread (the runtime's primary
// context of the current device, unless the caller made another current).
// Device addresses of the library's __device__ variables belong to one
// context: cudaDeviceReset or another context gives the same variable another
// address, so a cached address is keyed by this id.  False when no live
// context is current.  The driver calls are fetched through the runtime, so
// the library does not link libcuda directly.
inline bool current_context_id(unsigned long long* id) {
  typedef CUresult (*GetCurrentFn)(CUcontext*);
  typedef CUresult (*GetIdFn)(CUcontext, unsigned long long*);
  struct Fns {
    GetCurrentFn get_current = nullptr;
    GetIdFn get_id = nullptr;
  };
  static const Fns fns = [] {   // looked up once, thread-safely
    Fns f;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      f.get_current = reinterpret_cast<GetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      f.get_id = reinterpret_cast<GetIdFn>(p);
    return f;
  }();
  if (fns.get_current == nullptr || fns.get_id == nullptr) return false;
  CUcontext ctx = nullptr;
  if (fns.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return fns.get_id(ctx, id) == CUDA_SUCCESS;
}

// Device status codes written by kernels (same values as fa_status).
enum : int {
  kDevOk = 0,
  kDevInvalidArg = 1,
  kDevTimeout = 5,
  kDevBadBlockTable = 6,
  kDevDebugCheck = 7
};

// Debug builds (-DFA_DEBUG: libfa_gb300_debug.so) check each global store's
// index against the size of the buffer the kernel was given; a failed check
// records kDevDebugCheck in the status word and the store is skipped instead
// of landing outside the buffer.  In the normal build the check is the
// constant true and neither operand is evaluated.
#ifdef FA_DEBUG
#define FA_IN_BOUNDS(idx, limit, status)                     \
  (((size_t)(idx) < (size_t)(limit)) ? true                  \
                                     : (atomicExch((status), kDevDebugCheck), false))
#else
#define FA_IN_BOUNDS(idx, limit, status) true
#endif

// Forward problem.  Dense BSHD when cu_q == nullptr; otherwise packed varlen
// (B = number of sequences, n/m = max lengths, token rows start at cu_q[b]).
struct FwdParams {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;          // may be null
  const int* cu_q;     // varlen only (device)
  const int* cu_k;     // varlen only (device)
  int B, H, Hkv, n, m, d, dv;
  int total_q, total_k;  // varlen: rows of the packed q/k tensors (0 if unknown)
  float scale;
  int causal;
  int* status;         // device status word
  // paged prefill (block_table != nullptr): k, v are caches [pages][Hkv][16][d],
  // seq_lens[b] keys per sequence, q packed by cu_q as for varlen
  const int* block_table = nullptr;
  const int* seq_lens = nullptr;
  int max_blocks = 0;
  int num_pages = 0;
  // e4m3 operands (q, k, v hold x / descale), bf16 output
  int fp8 = 0;
  float q_descale = 1.f, k_descale = 1.f, v_descale = 1.f;
};

struct DecodeParams {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int* block_table;
  const int* seq_lens;
  int num_seqs, H, Hkv, d, dv, page_size, num_pages, max_blocks, num_splits;
  float scale;
  float* part_m;       // [S][H][X]
  float* part_l;       // [S][H][X]
  float* part_o;       // [S][H][X][dv]
  int* status;
  // fused form only: per (sequence, kv head) ticket counters, zero between
  // calls, and the outputs the merging split writes
  int* tickets = nullptr;
  void* o = nullptr;   // bf16 [S][H][dv]
  float* lse = nullptr;
};

struct CombineParams {
  const float* part_m;
  const float* part_l;
  const float* part_o;
  void* o;             // bf16 [S][H][dv]
  float* lse;          // [S][H], may be null
  int num_seqs, H, num_splits, dv;
};

struct GatherParams {
  const void* k_cache;
  const void* v_cache;
  const int* block_table;
  const int* seq_lens;
  void* k_out;         // bf16 [S][max_blocks * 16][Hkv][128]
  void* v_out;
  int num_seqs, Hkv, num_pages, max_blocks, num_splits;
  int* status;
};

cudaError_t launch_fwd_f32(const FwdParams& p, cudaStream_t stream);
cudaError_t launch_fwd_bf16(const FwdParams& p, cudaStream_t stream, const char** why);
// fused: partials and merge in one launch (p.tickets, p.o, p.lse set)
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream, bool fused);
cudaError_t launch_decode_partials(const DecodeParams& p, cudaStream_t stream);
// behind_partials: launched right after launch_decode_partials on the same
// stream, as a programmatic dependent of it
cudaError_t launch_split_combine(const CombineParams& p, cudaStream_t stream,
                                 bool behind_partials = false);
cudaError_t launch_decode_gather(const GatherParams& p, cudaStream_t stream);

}  // namespace fa
