// C ABI of libfa_gb300.so: argument validation, workspace carving, the device
// status word and error reporting.  Every entry point is declared and
// documented in include/fa.h; the kernels live in the other translation units.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace {

thread_local char g_err[512] = "";

fa_status fail(fa_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return st;
}

fa_status cuda_fail(cudaError_t e, const char* what) {
  return fail(FA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// One status word per device, in the library's own device memory: kernels
// record timeouts and bad block-table ids there instead of faulting.
__device__ int g_device_status = 0;

// Its device address belongs to the CUDA context the library's module is
// loaded in: after cudaDeviceReset, or in a context the caller created
// itself, the same variable has another address.  Addresses are therefore
// cached per context id (a few contexts at most), never per device ordinal.
constexpr int kMaxContexts = 64;
struct CtxAddr {
  unsigned long long ctx;
  int* ptr;
};
CtxAddr g_status_cache[kMaxContexts] = {};
int g_status_next = 0;
std::mutex g_status_mutex;

fa_status status_ptr(int** out) {
  std::lock_guard<std::mutex> lock(g_status_mutex);
  unsigned long long ctx = 0;
  if (fa::current_context_id(&ctx)) {
    for (const CtxAddr& c : g_status_cache)
      if (c.ptr != nullptr && c.ctx == ctx) {
        *out = c.ptr;
        return FA_OK;
      }
  }
  // not seen yet (or no context bound to this thread: the lookup below binds
  // the runtime's primary context of the current device)
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_device_status);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
  if (fa::current_context_id(&ctx)) {   // else (no context ids) look it up every call
    g_status_cache[g_status_next] = CtxAddr{ctx, static_cast<int*>(p)};
    g_status_next = (g_status_next + 1) % kMaxContexts;
  }
  *out = static_cast<int*>(p);
  return FA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

fa_status check_dense(const void* q, const void* k, const void* v, const void* o, const float* lse,
                      int B, int H, int Hkv, int n, int m, int d, int dv, int causal,
                      const char* fn) {
  if (B < 0 || n < 0 || m < 0) return fail(FA_ERR_INVALID_ARG, "%s: negative size", fn);
  if (H <= 0 || Hkv <= 0 || H % Hkv != 0)
    return fail(FA_ERR_INVALID_ARG, "%s: H=%d Hkv=%d (need H %% Hkv == 0)", fn, H, Hkv);
  if (d <= 0 || dv <= 0) return fail(FA_ERR_INVALID_ARG, "%s: d=%d dv=%d", fn, d, dv);
  if (causal != 0 && causal != 1) return fail(FA_ERR_INVALID_ARG, "%s: causal=%d", fn, causal);
  const bool empty_out = (B == 0 || n == 0);
  if (!empty_out && (q == nullptr || o == nullptr))
    return fail(FA_ERR_INVALID_ARG, "%s: null q/o", fn);
  if (!empty_out && m > 0 && (k == nullptr || v == nullptr))
    return fail(FA_ERR_INVALID_ARG, "%s: null k/v", fn);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(FA_ERR_INVALID_ARG, "%s: pointers must be 16-byte aligned (lse 4-byte)", fn);
  return FA_OK;
}

// Dense layouts: the kernels form token rows b*n + i and b*m + j, and the LSE
// stride H*n, in 32-bit ints.
fa_status check_rows(int B, int H, int n, int m, const char* fn) {
  const long long lim = 2147483647LL;
  if ((long long)B * n > lim || (long long)B * m > lim || (long long)H * n > lim)
    return fail(FA_ERR_UNSUPPORTED, "%s: B*n, B*m and H*n must stay below 2^31", fn);
  return FA_OK;
}

}  // namespace

// Shared with the other C-ABI translation units (same error text and status word).
namespace fa {
fa_status api_fail(fa_status st, const char* msg) { return fail(st, "%s", msg); }
fa_status api_status_ptr(int** out) { return status_ptr(out); }
}  // namespace fa

extern "C" {

const char* fa_last_error(void) { return g_err; }

fa_status fa_get_device_status(void* stream, int* status) {
  if (status == nullptr) return fail(FA_ERR_INVALID_ARG, "fa_get_device_status: null status");
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int* sp = nullptr;
  fa_status st = status_ptr(&sp);
  if (st != FA_OK) return st;
  int value = 0;
  e = cudaMemcpy(&value, sp, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read device status");
  const int zero = 0;
  e = cudaMemcpy(sp, &zero, sizeof(int), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "clear device status");
  *status = value;
  return FA_OK;
}

fa_status fa_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H, int Hkv, int n, int m, int d, int dv, float scale, int causal,
                     void* stream) {
  fa_status st = check_dense(q, k, v, o, lse, B, H, Hkv, n, m, d, dv, causal, "fa_forward");
  if (st != FA_OK) return st;
  if (!(scale > 0.f) || scale == INFINITY)
    return fail(FA_ERR_INVALID_ARG, "fa_forward: scale must be positive and finite");
  if (!(d == dv && (d == 64 || d == 128)))
    return fail(FA_ERR_UNSUPPORTED, "fa_forward: d=%d dv=%d (supported: d == dv in {64, 128})", d,
                dv);
  if ((st = check_rows(B, H, n, m, "fa_forward")) != FA_OK) return st;
  if (B == 0 || n == 0) return FA_OK;
  int* sp = nullptr;
  if ((st = status_ptr(&sp)) != FA_OK) return st;
  fa::FwdParams p{q, k, v, o, lse, nullptr, nullptr, B, H, Hkv, n, m, d, dv, 0, 0, scale, causal,
                  sp};
  const char* why = nullptr;
  cudaError_t e = fa::launch_fwd_bf16(p, static_cast<cudaStream_t>(stream), &why);
  if (e != cudaSuccess) return cuda_fail(e, why ? why : "fa_forward launch");
  return FA_OK;
}

fa_status fa_forward_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                         int H, int Hkv, int n, int m, int d, int dv, float scale,
                         float q_descale, float k_descale, float v_descale, int causal,
                         void* stream) {
  fa_status st = check_dense(q, k, v, o, lse, B, H, Hkv, n, m, d, dv, causal, "fa_forward_fp8");
  if (st != FA_OK) return st;
  if (!(scale > 0.f) || scale == INFINITY)
    return fail(FA_ERR_INVALID_ARG, "fa_forward_fp8: scale must be positive and finite");
  if (!(q_descale > 0.f) || !(k_descale > 0.f) || !(v_descale > 0.f) || q_descale == INFINITY ||
      k_descale == INFINITY || v_descale == INFINITY)
    return fail(FA_ERR_INVALID_ARG, "fa_forward_fp8: descale factors must be positive and finite");
  if (!(d == 128 && dv == 128))
    return fail(FA_ERR_UNSUPPORTED, "fa_forward_fp8: d=%d dv=%d (supported: 128)", d, dv);
  if ((st = check_rows(B, H, n, m, "fa_forward_fp8")) != FA_OK) return st;
  if (B == 0 || n == 0) return FA_OK;
  int* sp = nullptr;
  if ((st = status_ptr(&sp)) != FA_OK) return st;
  fa::FwdParams p{q, k, v, o, lse, nullptr, nullptr, B, H, Hkv, n, m, d, dv, 0, 0, scale, causal,
                  sp};
  p.fp8 = 1;
  p.q_descale = q_descale;
  p.k_descale = k_descale;
  p.v_descale = v_descale;
  const char* why = nullptr;
  cudaError_t e = fa::launch_fwd_bf16(p, static_cast<cudaStream_t>(stream), &why);
  if (e != cudaSuccess) return cuda_fail(e, why ? why : "fa_forward_fp8 launch");
  return FA_OK;
}

fa_status fa_forward_f32(const float* q, const float* k, const float* v, float* o, float* lse,
                         int B, int H, int Hkv, int n, int m, int d, int dv, float scale,
                         int causal, void* stream) {
  fa_status st = check_dense(q, k, v, o, lse, B, H, Hkv, n, m, d, dv, causal, "fa_forward_f32");
  if (st != FA_OK) return st;
  // the fp32 kernel takes the row max of the unscaled scores: a non-positive
  // scale would turn it into a minimum
  if (!(scale > 0.f) || scale == INFINITY)
    return fail(FA_ERR_INVALID_ARG, "fa_forward_f32: scale must be positive and finite");
  if (!((d == 64 || d == 128) && (dv == 64 || dv == 128)))
    return fail(FA_ERR_UNSUPPORTED, "fa_forward_f32: d=%d dv=%d (supported: 64, 128)", d, dv);
  // one CTA row block per (query block, head, batch): grid y and z hold H and B
  if (H > 65535 || B > 65535)
    return fail(FA_ERR_UNSUPPORTED, "fa_forward_f32: H=%d B=%d (at most 65535 each)", H, B);
  if (B == 0 || n == 0) return FA_OK;
  int* sp = nullptr;
  if ((st = status_ptr(&sp)) != FA_OK) return st;
  fa::FwdParams p{q, k, v, o, lse, nullptr, nullptr, B, H, Hkv, n, m, d, dv, 0, 0, scale, causal,
                  sp};
  cudaError_t e = fa::launch_fwd_f32(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fa_forward_f32 launch");
  return FA_OK;
}

fa_status fa_forward_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                            const int* cu_seqlens_q, const int* cu_seqlens_k, int num_seqs,
                            int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int H,
                            int Hkv, int d, int dv, float scale, int causal, void* stream) {
  if (num_seqs < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 || total_q < 0 || total_k < 0)
    return fail(FA_ERR_INVALID_ARG, "fa_forward_varlen: negative size");
  if (!(scale > 0.f) || scale == INFINITY)
    return fail(FA_ERR_INVALID_ARG, "fa_forward_varlen: scale must be positive and finite");
  if (num_seqs > 0 && (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr))
    return fail(FA_ERR_INVALID_ARG, "fa_forward_varlen: null cu_seqlens");
  fa_status st = check_dense(q, k, v, o, lse, num_seqs, H, Hkv, max_seqlen_q, max_seqlen_k, d, dv,
                             0, "fa_forward_varlen");
  if (st != FA_OK) return st;
  if (causal != 0 && causal != 1)
    return fail(FA_ERR_INVALID_ARG, "fa_forward_varlen: causal=%d", causal);
  if (!(d == dv && (d == 64 || d == 128)))
    return fail(FA_ERR_UNSUPPORTED, "fa_forward_varlen: d=%d dv=%d (supported: d == dv in {64, 128})",
                d, dv);
  if (num_seqs == 0 || max_seqlen_q == 0 || total_q == 0) return FA_OK;
  int* sp = nullptr;
  if ((st = status_ptr(&sp)) != FA_OK) return st;
  fa::FwdParams p{q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, num_seqs, H, Hkv,
                  max_seqlen_q, max_seqlen_k, d, dv, total_q, total_k, scale, causal, sp};
  const char* why = nullptr;
  cudaError_t e = fa::launch_fwd_bf16(p, static_cast<cudaStream_t>(stream), &why);
  if (e != cudaSuccess) return cuda_fail(e, why ? why : "fa_forward_varlen launch");
  return FA_OK;
}

fa_status fa_paged_prefill(const void* q, const void* k_cache, const void* v_cache,
                           const int* block_table, const int* seq_lens, const int* cu_seqlens_q,
                           void* o, float* lse, int num_seqs, int total_q, int max_seqlen_q,
                           int H, int Hkv, int d, int dv, int page_size, int num_pages,
                           int max_blocks_per_seq, float scale, int causal, void* stream) {
  const char* fn = "fa_paged_prefill";
  if (num_seqs < 0 || total_q < 0 || max_seqlen_q < 0 || num_pages < 0 || max_blocks_per_seq < 0)
    return fail(FA_ERR_INVALID_ARG, "%s: negative size", fn);
  if (H <= 0 || Hkv <= 0 || H % Hkv != 0)
    return fail(FA_ERR_INVALID_ARG, "%s: H=%d Hkv=%d (need H %% Hkv == 0)", fn, H, Hkv);
  if (causal != 0 && causal != 1) return fail(FA_ERR_INVALID_ARG, "%s: causal=%d", fn, causal);
  if (!(scale > 0.f) || scale == INFINITY)
    return fail(FA_ERR_INVALID_ARG, "%s: scale must be positive and finite", fn);
  if (!(d == dv && (d == 64 || d == 128)))
    return fail(FA_ERR_UNSUPPORTED, "%s: d=%d dv=%d (supported: d == dv in {64, 128})", fn, d, dv);
  if (page_size != 16) return fail(FA_ERR_UNSUPPORTED, "%s: page_size=%d (supported: 16)", fn, page_size);
  if (num_seqs == 0 || total_q == 0 || max_seqlen_q == 0) return FA_OK;
  if (q == nullptr || o == nullptr || k_cache == nullptr || v_cache == nullptr ||
      block_table == nullptr || seq_lens == nullptr || cu_seqlens_q == nullptr)
    return fail(FA_ERR_INVALID_ARG, "%s: null pointer", fn);
  if (num_pages == 0 || max_blocks_per_seq == 0)
    return fail(FA_ERR_INVALID_ARG, "%s: empty page pool or block table", fn);
  if ((long long)num_pages * Hkv * 16 > 0x7fffffffLL)
    return fail(FA_ERR_UNSUPPORTED, "%s: page pool too large", fn);
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(block_table) & 3u) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u) || (reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3u))
    return fail(FA_ERR_INVALID_ARG, "%s: misaligned pointer", fn);
  int* sp = nullptr;
  fa_status st = status_ptr(&sp);
  if (st != FA_OK) return st;
  fa::FwdParams p{q, k_cache, v_cache, o, lse, cu_seqlens_q, nullptr, num_seqs, H, Hkv,
                  max_seqlen_q, 0, d, dv, total_q, 0, scale, causal, sp};
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.max_blocks = max_blocks_per_seq;
  p.num_pages = num_pages;
  const char* why = nullptr;
  cudaError_t e = fa::launch_fwd_bf16(p, static_cast<cudaStream_t>(stream), &why);
  if (e != cudaSuccess) return cuda_fail(e, why ? why : "fa_paged_prefill launch");
  return FA_OK;
}

static size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t fa_paged_decode_workspace_size(int num_seqs, int H, int dv, int num_splits) {
  if (num_seqs < 0 || H <= 0 || dv <= 0 || num_splits <= 0) return 0;
  const size_t tri = (size_t)num_seqs * H * num_splits;
  // the fused form's ticket counters first (one per (sequence, head) bounds
  // the one per (sequence, kv head) it uses; at a fixed offset, so zeroed
  // once they serve every split count), then partial m, l and o
  return round256((size_t)num_seqs * H * sizeof(int)) + 2 * round256(tri * sizeof(float)) +
         round256(tri * dv * sizeof(float));
}

}  // extern "C"

namespace {

// Argument checks and workspace carving shared by the two decode entries.
fa_status decode_setup(const char* fn, const void* q, const void* k_cache, const void* v_cache,
                       const int* block_table, const int* seq_lens, void* o, float* lse,
                       int num_seqs, int H, int Hkv, int d, int dv, int page_size, int num_pages,
                       int max_blocks_per_seq, int num_splits, float scale, void* workspace,
                       size_t workspace_bytes, fa::DecodeParams* p, bool* nothing) {
  *nothing = false;
  if (num_seqs < 0 || num_pages < 0 || max_blocks_per_seq < 0)
    return fail(FA_ERR_INVALID_ARG, "%s: negative size", fn);
  if (H <= 0 || Hkv <= 0 || H % Hkv != 0)
    return fail(FA_ERR_INVALID_ARG, "%s: H=%d Hkv=%d (need H %% Hkv == 0)", fn, H, Hkv);
  if (num_splits < 1 || num_splits > 64)
    return fail(FA_ERR_INVALID_ARG, "%s: num_splits=%d outside [1, 64]", fn, num_splits);
  if (!(scale > 0.f) || scale == INFINITY)
    return fail(FA_ERR_INVALID_ARG, "%s: scale must be positive and finite", fn);
  if (d != 128 || dv != 128)
    return fail(FA_ERR_UNSUPPORTED, "%s: d=%d dv=%d (supported: 128)", fn, d, dv);
  if (page_size != 16) return fail(FA_ERR_UNSUPPORTED, "%s: page_size=%d (supported: 16)", fn, page_size);
  if (H / Hkv > 16) return fail(FA_ERR_UNSUPPORTED, "%s: H/Hkv=%d > 16", fn, H / Hkv);
  if (num_seqs == 0) {
    *nothing = true;
    return FA_OK;
  }
  if (q == nullptr || o == nullptr || block_table == nullptr || seq_lens == nullptr ||
      k_cache == nullptr || v_cache == nullptr)
    return fail(FA_ERR_INVALID_ARG, "%s: null pointer", fn);
  if (num_pages == 0 || max_blocks_per_seq == 0)
    return fail(FA_ERR_INVALID_ARG, "%s: empty page pool or block table", fn);
  // page rows (page * Hkv + head) * 16 and the units (sequence, head, split) are 32-bit
  if ((long long)num_pages * Hkv * 16 > 0x7fffffffLL ||
      (long long)num_seqs * H * num_splits > 0x7fffffffLL)
    return fail(FA_ERR_UNSUPPORTED, "%s: page pool or sequences x heads x splits too large", fn);
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(block_table) & 3u) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return fail(FA_ERR_INVALID_ARG, "%s: misaligned pointer", fn);
  const size_t need = fa_paged_decode_workspace_size(num_seqs, H, dv, num_splits);
  if (workspace == nullptr || workspace_bytes < need ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(FA_ERR_WORKSPACE, "%s: workspace %p of %zu bytes (need %zu, 256-byte aligned)", fn,
                workspace, workspace_bytes, need);
  int* sp = nullptr;
  fa_status st = status_ptr(&sp);
  if (st != FA_OK) return st;
  const size_t tri = (size_t)num_seqs * H * num_splits;
  char* ws = static_cast<char*>(workspace);
  int* tickets = reinterpret_cast<int*>(ws);
  ws += round256((size_t)num_seqs * H * sizeof(int));
  float* part_m = reinterpret_cast<float*>(ws);
  float* part_l = reinterpret_cast<float*>(ws + round256(tri * sizeof(float)));
  float* part_o = reinterpret_cast<float*>(ws + 2 * round256(tri * sizeof(float)));
  *p = fa::DecodeParams{q, k_cache, v_cache, block_table, seq_lens, num_seqs, H, Hkv, d, dv,
                        page_size, num_pages, max_blocks_per_seq, num_splits, scale,
                        part_m, part_l, part_o, sp};
  p->tickets = tickets;
  p->o = o;
  p->lse = lse;
  return FA_OK;
}

}  // namespace

extern "C" {

fa_status fa_paged_decode(const void* q, const void* k_cache, const void* v_cache,
                          const int* block_table, const int* seq_lens, void* o, float* lse,
                          int num_seqs, int H, int Hkv, int d, int dv, int page_size,
                          int num_pages, int max_blocks_per_seq, int num_splits, float scale,
                          void* workspace, size_t workspace_bytes, void* stream) {
  fa::DecodeParams p{};
  bool nothing = false;
  fa_status st = decode_setup("fa_paged_decode", q, k_cache, v_cache, block_table, seq_lens, o,
                              lse, num_seqs, H, Hkv, d, dv, page_size, num_pages,
                              max_blocks_per_seq, num_splits, scale, workspace, workspace_bytes,
                              &p, &nothing);
  if (st != FA_OK || nothing) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = fa::launch_decode_partials(p, s);
  if (e != cudaSuccess) return cuda_fail(e, "fa_paged_decode partials launch");
  fa::CombineParams c{p.part_m, p.part_l, p.part_o, o, lse, num_seqs, H, num_splits, dv};
  e = fa::launch_split_combine(c, s, true);
  if (e != cudaSuccess) return cuda_fail(e, "fa_paged_decode combine launch");
  return FA_OK;
}

fa_status fa_paged_decode_fused(const void* q, const void* k_cache, const void* v_cache,
                                const int* block_table, const int* seq_lens, void* o, float* lse,
                                int num_seqs, int H, int Hkv, int d, int dv, int page_size,
                                int num_pages, int max_blocks_per_seq, int num_splits, float scale,
                                void* workspace, size_t workspace_bytes, void* stream) {
  fa::DecodeParams p{};
  bool nothing = false;
  fa_status st = decode_setup("fa_paged_decode_fused", q, k_cache, v_cache, block_table,
                              seq_lens, o, lse, num_seqs, H, Hkv, d, dv, page_size, num_pages,
                              max_blocks_per_seq, num_splits, scale, workspace, workspace_bytes,
                              &p, &nothing);
  if (st != FA_OK || nothing) return st;
  cudaError_t e = fa::launch_decode(p, static_cast<cudaStream_t>(stream), true);
  if (e != cudaSuccess) return cuda_fail(e, "fa_paged_decode_fused launch");
  return FA_OK;
}

fa_status fa_paged_gather(const void* k_cache, const void* v_cache, const int* block_table,
                          const int* seq_lens, void* k_out, void* v_out, int num_seqs, int Hkv,
                          int d, int page_size, int num_pages, int max_blocks_per_seq,
                          int num_splits, void* stream) {
  const char* fn = "fa_paged_gather";
  if (num_seqs < 0 || num_pages < 0 || max_blocks_per_seq < 0)
    return fail(FA_ERR_INVALID_ARG, "%s: negative size", fn);
  if (Hkv <= 0) return fail(FA_ERR_INVALID_ARG, "%s: Hkv=%d", fn, Hkv);
  if (num_splits < 1 || num_splits > 64)
    return fail(FA_ERR_INVALID_ARG, "%s: num_splits=%d outside [1, 64]", fn, num_splits);
  if (d != 128) return fail(FA_ERR_UNSUPPORTED, "%s: d=%d (supported: 128)", fn, d);
  if (page_size != 16) return fail(FA_ERR_UNSUPPORTED, "%s: page_size=%d (supported: 16)", fn, page_size);
  if (num_seqs == 0) return FA_OK;
  if (k_cache == nullptr || v_cache == nullptr || block_table == nullptr || seq_lens == nullptr ||
      k_out == nullptr || v_out == nullptr)
    return fail(FA_ERR_INVALID_ARG, "%s: null pointer", fn);
  if (num_pages == 0 || max_blocks_per_seq == 0)
    return fail(FA_ERR_INVALID_ARG, "%s: empty page pool or block table", fn);
  if ((long long)num_pages * Hkv * 16 > 0x7fffffffLL ||
      (long long)num_seqs * Hkv * num_splits > 0x7fffffffLL)
    return fail(FA_ERR_UNSUPPORTED, "%s: page pool or sequences x heads x splits too large", fn);
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_out) || !aligned16(v_out) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return fail(FA_ERR_INVALID_ARG, "%s: misaligned pointer", fn);
  int* sp = nullptr;
  fa_status st = status_ptr(&sp);
  if (st != FA_OK) return st;
  fa::GatherParams p{k_cache, v_cache, block_table, seq_lens, k_out, v_out,
                     num_seqs, Hkv, num_pages, max_blocks_per_seq, num_splits, sp};
  cudaError_t e = fa::launch_decode_gather(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fa_paged_gather launch");
  return FA_OK;
}

fa_status fa_split_combine(const float* part_m, const float* part_l, const float* part_o, void* o,
                           float* lse, int num_seqs, int H, int num_splits, int dv, void* stream) {
  const char* fn = "fa_split_combine";
  if (num_seqs < 0 || H <= 0) return fail(FA_ERR_INVALID_ARG, "%s: bad sizes", fn);
  if (num_splits < 1 || num_splits > 64)
    return fail(FA_ERR_INVALID_ARG, "%s: num_splits=%d outside [1, 64]", fn, num_splits);
  if (dv <= 0 || dv % 4 != 0 || dv > 256)
    return fail(FA_ERR_UNSUPPORTED, "%s: dv=%d (need dv %% 4 == 0, dv <= 256)", fn, dv);
  if ((long long)num_seqs * H > 0x7fffffffLL)
    return fail(FA_ERR_UNSUPPORTED, "%s: sequences x heads too large", fn);
  if (num_seqs == 0) return FA_OK;
  if (part_m == nullptr || part_l == nullptr || part_o == nullptr || o == nullptr)
    return fail(FA_ERR_INVALID_ARG, "%s: null pointer", fn);
  if (!aligned16(part_o) || (reinterpret_cast<uintptr_t>(o) & 7u) ||
      (reinterpret_cast<uintptr_t>(part_m) & 3u) || (reinterpret_cast<uintptr_t>(part_l) & 3u) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(FA_ERR_INVALID_ARG, "%s: misaligned pointer", fn);
  fa::CombineParams c{part_m, part_l, part_o, o, lse, num_seqs, H, num_splits, dv};
  cudaError_t e = fa::launch_split_combine(c, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fa_split_combine launch");
  return FA_OK;
}

}  // extern "C"
