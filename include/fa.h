/*
 * fa.h — C ABI of the GB300 (sm_103a) tiled online-softmax attention library
 * (libfa_gb300.so).
 *
 * What it computes.  Exact scaled-dot-product attention
 *     O = softmax(scale * Q K^T) V,   row-wise softmax,
 * with Q n×d, K m×d, V m×dv and O n×dv per (batch, head)
 * ("手搓 Attention：从三行循环到看懂 FlashAttention", §1).  The kernels never
 * form the n×m score matrix in memory: they stream K/V tiles and keep, per
 * query row, a running maximum m, a running sum l and an accumulator acc that
 * are rescaled by alpha = exp(m_old - m_new) whenever the maximum grows
 * (same page, §7 version 4; "S12 FlashAttention", 解法).  The log-sum-exp
 * LSE = m + ln(l) (natural log, over the SCALED scores) is returned beside O.
 *
 * Conventions shared by every entry point.
 *   - Pointers are DEVICE pointers owned by the caller, unless a parameter
 *     says otherwise.  The library never allocates device memory for a call;
 *     decode takes its split scratch from a caller-provided workspace.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and returns as soon as its launches are queued.
 *   - Arguments are validated before anything is launched; on a bad argument
 *     the call returns a non-zero fa_status and launches nothing.  The text of
 *     the last failure on the calling thread is returned by fa_last_error().
 *   - Problems that only the device can see (a block-table id out of range,
 *     a pipeline wait that exceeded its time limit) set a device status word
 *     instead of faulting; the affected outputs are left unspecified.
 *     fa_get_device_status() synchronises the stream and reads and clears it.
 *   - Layouts are dense row-major.  "BSHD" means [batch][token][head][dim].
 *   - Grouped heads: query head h reads kv head h / (H / Hkv); H % Hkv == 0.
 *   - bf16 values are IEEE bfloat16 bit patterns (uint16 storage); outputs O
 *     are rounded to bf16 with round-to-nearest-even; LSE is float32.
 *   - A query row that sees no key gets O = 0 and LSE = -inf.
 *   - Causal: key j is visible to query i iff j <= i + (m - n) (0-based):
 *     the n queries are the last n of the m key positions.  For n == m this
 *     is "query i sees the keys up to i"; for n > m the first n - m queries
 *     see no key (O = 0, LSE = -inf).  Varlen applies it per sequence.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,   /* null pointer, negative size, H % Hkv != 0, misaligned pointer */
    FA_ERR_UNSUPPORTED = 2,   /* valid but not implemented: d/dv/page_size outside the supported set,
                                 no sm_103a device */
    FA_ERR_WORKSPACE = 3,     /* workspace pointer null or smaller than the size query returns */
    FA_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed; fa_last_error() has the text */
    FA_ERR_TIMEOUT = 5,       /* device status: a pipeline wait exceeded its limit */
    FA_ERR_BAD_BLOCK_TABLE = 6, /* device status: a block-table id outside [0, num_pages) */
    FA_ERR_DEBUG_CHECK = 7    /* device status, debug build (libfa_gb300_debug.so) only: a
                                 kernel's output index left the buffer it was given; the store
                                 was skipped.  Never set by the normal build. */
} fa_status;

/*
 * fa_forward — bf16 attention forward, dense batch.
 * Passage: "手搓 Attention" §1 (shapes and scale) and §7 version 4 (the
 * recurrence); "S12 FlashAttention", 解法; whole causal tiles above the
 * diagonal are skipped ("手搓 Attention" §6 and §7).
 *
 *   q    bf16 [B][n][H][d]       (BSHD)
 *   k    bf16 [B][m][Hkv][d]
 *   v    bf16 [B][m][Hkv][dv]
 *   o    bf16 [B][n][H][dv]      written
 *   lse  fp32 [B][H][n]          written (may be NULL: not written)
 *   scale  multiplies Q K^T; must be positive and finite (pass 1/sqrt(d)
 *          for the usual attention)
 *   causal 0 or 1
 * Non-finite inputs stay in their own batch element: the last K/V tile of an
 * element whose m is not a multiple of the tile reads zeros past its last row
 * (never the next element's rows, whose inf or NaN would otherwise turn the
 * masked keys' zero weights into NaN: 0 * inf = NaN).
 * Supported: d == dv, d in {64, 128}; pointers 16-byte aligned; n, m >= 0;
 * B*n, B*m and H*n below 2^31 (token rows and the LSE stride are 32-bit).
 * Computes S = Q K^T and P V on the tcgen05 tensor cores (bf16 operands,
 * fp32 accumulation in tensor memory); P is rounded to bf16 before P V.
 */
fa_status fa_forward(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int H, int Hkv, int n, int m, int d, int dv,
                     float scale, int causal, void* stream);

/*
 * fa_forward_fp8 — attention forward with e4m3 (FP8) operands and per-tensor
 * descale factors: the values are q[i] * q_descale, k[j] * k_descale,
 * v[j] * v_descale.  Same shapes, layouts and semantics as fa_forward; o is
 * bf16, lse fp32 (of the descaled scores).  The pages name FP8 only as a
 * later FlashAttention feature ("S12 FlashAttention", 生产实践); the
 * recurrence is unchanged: S = Q K^T and P V run on the tcgen05 tensor cores
 * in kind::f8f6f4 with fp32 accumulation, and P is rounded to e4m3 (it lies
 * in [0, 256] under the lazy rescale, inside e4m3's range) before P V.
 *   q, k, v   e4m3 bytes [B][n][H][d], [B][m][Hkv][d], [B][m][Hkv][dv]
 *   descales  positive finite fp32
 * Supported: d == dv == 128; B*n, B*m and H*n below 2^31.
 */
fa_status fa_forward_fp8(const void* q, const void* k, const void* v, void* o, float* lse,
                         int B, int H, int Hkv, int n, int m, int d, int dv, float scale,
                         float q_descale, float k_descale, float v_descale, int causal,
                         void* stream);

/*
 * fa_forward_f32 — fp32 attention forward, dense batch; same shapes, layouts
 * and semantics as fa_forward with every tensor in float32.
 * Passage: "手搓 Attention" §1 (shapes and scale), §4 version 2 (subtract the
 * row maximum before exp; in fp32 that keeps hot scores of several hundred
 * finite and within a few 1e-6 of float64) and §7 version 4 (the recurrence).
 * Arithmetic is IEEE fp32 on the CUDA cores (no TF32); each score is carried
 * as a compensated (hi, lo) pair so that exp(s - m) keeps fp32 relative
 * accuracy when the scores are in the hundreds.
 *   scale  must be positive and finite, as for fa_forward (the row maximum is
 *          taken on the unscaled scores, which is the scaled maximum only for
 *          a positive scale); anything else returns FA_ERR_INVALID_ARG
 * Supported: d, dv in {64, 128}; pointers 16-byte aligned; H, B <= 65535.
 */
fa_status fa_forward_f32(const float* q, const float* k, const float* v, float* o, float* lse,
                         int B, int H, int Hkv, int n, int m, int d, int dv,
                         float scale, int causal, void* stream);

/*
 * fa_forward_varlen — bf16 attention forward over packed sequences of
 * different lengths.  Sequence s owns query tokens [cu_seqlens_q[s],
 * cu_seqlens_q[s+1]) and key tokens [cu_seqlens_k[s], cu_seqlens_k[s+1]).
 * Passage: each sequence is its own attention problem ("手搓 Attention" §1),
 * computed by the same recurrence (§7 version 4; "S12 FlashAttention", 解法)
 * over that sequence's K/V tiles only; a sequence whose length is not a
 * multiple of the tile ends on a partly masked tile, and rows whose first
 * tiles are fully masked take the guard of "S12 FlashAttention", 实现.
 *
 *   q    bf16 [total_q][H][d],  k bf16 [total_k][Hkv][d],  v bf16 [total_k][Hkv][dv]
 *   o    bf16 [total_q][H][dv]  written
 *   lse  fp32 [H][total_q] written (may be NULL)
 *   cu_seqlens_q, cu_seqlens_k  int32 [num_seqs + 1], DEVICE pointers,
 *        non-decreasing, starting at 0, ending at total_q / total_k
 *   total_q, total_k  rows of the packed q (and o) and k/v buffers; the
 *        kernels never read or write a row outside them (a sequence whose
 *        offsets exceed them is skipped and sets FA_ERR_INVALID_ARG in the
 *        device status word)
 *   max_seqlen_q, max_seqlen_k  upper bounds of the per-sequence lengths
 *        (sizes the launch grid; a larger value only launches idle blocks)
 * Supported as fa_forward; causal uses each sequence's own q and k lengths.
 * Non-finite values stay in their own sequence: the V rows past a sequence's
 * end in its last K/V tile (the next sequence's rows) are zeroed in shared
 * memory before P V, as the paged paths do with the rows past a sequence's
 * end in its last page.
 */
fa_status fa_forward_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                            const int* cu_seqlens_q, const int* cu_seqlens_k, int num_seqs,
                            int total_q, int total_k, int max_seqlen_q, int max_seqlen_k,
                            int H, int Hkv, int d, int dv, float scale, int causal, void* stream);

/*
 * fa_paged_prefill — bf16 attention for several new query tokens per
 * sequence against that sequence's paged keys (chunked prefill).
 * Passage: "S12 FlashAttention", 它还解锁了什么 (the tiles the recurrence walks
 * need not be contiguous: each can be fetched through a block table) and 实现
 * (logical page p holds min(page_size, seq_len - p*page_size) valid tokens).
 *
 *   q            bf16 [total_q][H][d], sequence s owns rows
 *                [cu_seqlens_q[s], cu_seqlens_q[s+1])
 *   k_cache      bf16 [num_pages][Hkv][page_size][d]
 *   v_cache      bf16 [num_pages][Hkv][page_size][dv]
 *   block_table  int32 [num_seqs][max_blocks_per_seq]: logical -> physical page
 *   seq_lens     int32 [num_seqs]: keys of sequence s (its cached context and
 *                its new tokens), 0 <= seq_lens[s] <= max_blocks_per_seq*page_size
 *   cu_seqlens_q int32 [num_seqs + 1], non-decreasing from 0 to total_q
 *   o            bf16 [total_q][H][dv] written
 *   lse          fp32 [H][total_q]     written (may be NULL)
 *   max_seqlen_q upper bound of the per-sequence query counts
 *   causal       0 or 1: with 1 the n_s queries of sequence s are the last n_s
 *                of its seq_lens[s] positions (query i sees keys j <= i +
 *                seq_lens[s] - n_s)
 * All of K/V is read through TMA a page at a time on the tcgen05 path of
 * fa_forward.  Cache contents past seq_lens[s] in the last page are never
 * used, NaN included.  Page ids are range-checked on the device (an id
 * outside [0, num_pages) reads page 0 and sets FA_ERR_BAD_BLOCK_TABLE);
 * sequences whose query offsets fall outside total_q, or whose seq_lens[s]
 * falls outside [0, max_blocks_per_seq*page_size], are skipped (none of their
 * rows is written) and set FA_ERR_INVALID_ARG.
 * Supported: d == dv in {64, 128}, page_size == 16.
 */
fa_status fa_paged_prefill(const void* q, const void* k_cache, const void* v_cache,
                           const int* block_table, const int* seq_lens, const int* cu_seqlens_q,
                           void* o, float* lse, int num_seqs, int total_q, int max_seqlen_q,
                           int H, int Hkv, int d, int dv, int page_size, int num_pages,
                           int max_blocks_per_seq, float scale, int causal, void* stream);

/*
 * fa_paged_decode_workspace_size — bytes of workspace fa_paged_decode and
 * fa_paged_decode_fused need: the fused form's ticket words first (int32
 * [num_seqs][H], at the same offset for every split count), then the
 * per-split partial triples (m, l: fp32 [num_seqs][H][num_splits] each; o:
 * fp32 [num_seqs][H][num_splits][dv]), each array 256-byte aligned.
 * Passage: "S12 FlashAttention", 它还解锁了什么 and 练习 1 (flash-decoding:
 * each split of the keys leaves one (m, l, o) triple per query head, and the
 * merge reads them all).
 * Returns 0 on invalid sizes.
 */
size_t fa_paged_decode_workspace_size(int num_seqs, int H, int dv, int num_splits);

/*
 * fa_paged_decode — one query token per sequence against a paged KV cache,
 * split-KV ("flash-decoding"), grouped heads.
 * Passage: "S12 FlashAttention", 实现 (walk the block table; logical page p
 * holds min(page_size, seq_len - p*page_size) valid tokens), 组合 (block
 * table + grouped-head sharing + (m, l, o) in one loop), 它还解锁了什么 and
 * 练习 1 (split the keys across blocks, merge the (m, l, o) triples).
 *
 *   q            bf16 [num_seqs][H][d]
 *   k_cache      bf16 [num_pages][Hkv][page_size][d]
 *   v_cache      bf16 [num_pages][Hkv][page_size][dv]
 *   block_table  int32 [num_seqs][max_blocks_per_seq]: logical -> physical page
 *   seq_lens     int32 [num_seqs], 0 <= seq_lens[s] <= max_blocks_per_seq*page_size
 *   o            bf16 [num_seqs][H][dv]  written
 *   lse          fp32 [num_seqs][H]      written (may be NULL)
 *   num_splits   1..64: split x of a sequence with P pages covers logical
 *                pages [ceil(x*P/X), ceil((x+1)*P/X)); empty splits are allowed
 *   scale        positive and finite (else FA_ERR_INVALID_ARG)
 *   workspace    device scratch of at least fa_paged_decode_workspace_size()
 *                bytes, 256-byte aligned; the call writes the partials there
 *                and then merges them (fa_split_combine) on the same stream.
 * Tokens past seq_len in the last page are never used (their cache contents
 * may be anything, NaN included).  Page ids are range-checked on the device:
 * an id outside [0, num_pages) is skipped and sets FA_ERR_BAD_BLOCK_TABLE.  A
 * seq_lens[s] outside [0, max_blocks_per_seq*page_size] is treated as an
 * empty sequence (O = 0, LSE = -inf) and sets FA_ERR_INVALID_ARG.
 * Supported: d == dv == 128, page_size == 16, H / Hkv <= 16; num_pages*Hkv*16
 * and num_seqs*H*num_splits below 2^31.
 */
fa_status fa_paged_decode(const void* q, const void* k_cache, const void* v_cache,
                          const int* block_table, const int* seq_lens, void* o, float* lse,
                          int num_seqs, int H, int Hkv, int d, int dv, int page_size,
                          int num_pages, int max_blocks_per_seq, int num_splits, float scale,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_paged_decode_fused — fa_paged_decode in one launch.
 * Passage: "S12 FlashAttention", 接下来 (fuse the small-batch decode) and
 * 练习 1 (the split triples merge with the recurrence's rescale).
 *
 * Same arguments, layouts, supported sizes and device status as
 * fa_paged_decode, and the same O and LSE bits.  The merge runs inside the
 * decode launch: each (sequence, kv head, split) unit writes its triple,
 * then takes an atomic ticket of its (sequence, kv head); the unit that takes
 * the last ticket merges the triples of the group's query heads.  No unit
 * waits for another.
 *   workspace  as fa_paged_decode (the same size query).  Its ticket words
 *              must be zero before the first call that uses this workspace
 *              (cudaMemset the whole workspace to 0 once after allocating
 *              it); every call, also one that ends with FA_ERR_TIMEOUT,
 *              leaves them zero again.  Calls on one workspace must not
 *              overlap on the GPU.  (fa_paged_decode ignores the ticket
 *              words, so one workspace may serve both entries.)
 * After FA_ERR_TIMEOUT, O and LSE are undefined, as for fa_paged_decode.
 */
fa_status fa_paged_decode_fused(const void* q, const void* k_cache, const void* v_cache,
                                const int* block_table, const int* seq_lens, void* o, float* lse,
                                int num_seqs, int H, int Hkv, int d, int dv, int page_size,
                                int num_pages, int max_blocks_per_seq, int num_splits, float scale,
                                void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_paged_decode_noalloc — fa_paged_decode for callers that cannot allocate.
 * The pages have no counterpart for this call: it exists for library users.
 *
 * Some callers may not call cudaMalloc themselves: a plugin inside a host
 * framework that owns all device memory through its own allocator, or a
 * serving loop that must not allocate once it runs (cudaMalloc can
 * synchronise the device).  This entry point computes exactly what
 * fa_paged_decode computes (same kernels, same arguments minus the
 * workspace) and keeps its split partials in one fixed device array of
 * FA_NOALLOC_SCRATCH_BYTES that the library itself declares.  It allocates
 * nothing; the caller still owns and passes every input and output.
 *   - Every GPU that loads the library holds that array until the process ends.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and keeps it; make
 *     that first call before any stream capture.  The address is kept per
 *     CUDA context: after cudaDeviceReset the next call is again a first
 *     call (it looks the new address up), so make it outside a capture too.
 *   - A problem whose partials (fa_paged_decode_workspace_size) exceed the
 *     array is rejected with FA_ERR_WORKSPACE before anything is launched.
 *   - All calls share the array, which keeps the last call's contents.  A
 *     call that ends with the device status clear has rewritten every partial
 *     its merge read, so nothing needs clearing.  After FA_ERR_TIMEOUT some
 *     partials were not rewritten and the merge read the previous call's:
 *     that call's O and LSE are undefined.  Calls that overlap on the GPU
 *     (other streams, other threads) race on the array and corrupt each
 *     other: serialise them.
 * Arguments, layouts, supported sizes and device status as fa_paged_decode.
 */
#define FA_NOALLOC_SCRATCH_BYTES (16u << 20)
fa_status fa_paged_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                  const int* block_table, const int* seq_lens, void* o,
                                  float* lse, int num_seqs, int H, int Hkv, int d, int dv,
                                  int page_size, int num_pages, int max_blocks_per_seq,
                                  int num_splits, float scale, void* stream);

/*
 * fa_paged_gather — checking tool for the block-table walk of fa_paged_decode.
 * Passage: "S12 FlashAttention", 实现 (logical page p of sequence s is
 * physical page block_table[s][p] and holds min(page_size, seq_len -
 * p*page_size) valid tokens).
 *
 * Runs the decode's units (sequence, kv head, split) with the decode's split
 * page ranges, page lookups, tensor copies and shared-memory page layout, and
 * copies the K and V rows it gathers out to dense buffers instead of scoring
 * them, so a test can compare them bit for bit with a host gather.
 *   k_cache, v_cache, block_table, seq_lens, num_pages, max_blocks_per_seq,
 *   num_splits   as fa_paged_decode
 *   k_out, v_out bf16 [num_seqs][max_blocks_per_seq*page_size][Hkv][d],
 *                caller-owned: token t of sequence s is written to row
 *                s*max_blocks_per_seq*page_size + t for t < seq_lens[s]; other
 *                rows are not written.
 * Device status as fa_paged_decode (bad page ids, out-of-range seq_lens).
 * Supported: d == 128, page_size == 16; num_pages*Hkv*16 and
 * num_seqs*Hkv*num_splits below 2^31.
 */
fa_status fa_paged_gather(const void* k_cache, const void* v_cache, const int* block_table,
                          const int* seq_lens, void* k_out, void* v_out, int num_seqs, int Hkv,
                          int d, int page_size, int num_pages, int max_blocks_per_seq,
                          int num_splits, void* stream);

/*
 * fa_split_combine — merge per-split partial triples with the recurrence's
 * rescale rule ("S12 FlashAttention", 练习 1): for each (s, h)
 *     M = max_x m_x,  w_x = exp(m_x - M)  (w_x = 0 when m_x = -inf),
 *     l = sum_x w_x l_x,  O = sum_x w_x o_x / l,  LSE = M + ln l.
 *
 *   part_m, part_l  fp32 [num_seqs][H][num_splits]: m_x is the split's maximum
 *                   scaled score (natural units), l_x = sum exp(s_j - m_x)
 *   part_o          fp32 [num_seqs][H][num_splits][dv]: sum exp(s_j - m_x) V[j]
 *   o               bf16 [num_seqs][H][dv] written
 *   lse             fp32 [num_seqs][H] written (may be NULL)
 * An (s, h) whose splits are all empty gets O = 0 and LSE = -inf.
 * Supported: dv % 4 == 0, dv <= 256, 1 <= num_splits <= 64; num_seqs*H below 2^31.
 */
fa_status fa_split_combine(const float* part_m, const float* part_l, const float* part_o,
                           void* o, float* lse, int num_seqs, int H, int num_splits, int dv,
                           void* stream);

/*
 * fa_last_error — NUL-terminated description of the last non-OK status
 * returned on the calling thread ("" if none).  Owned by the library; valid
 * until the thread's next failing call.
 */
const char* fa_last_error(void);

/*
 * fa_get_device_status — synchronise `stream`, then read and clear the
 * device status word of the current device (FA_OK, FA_ERR_TIMEOUT,
 * FA_ERR_BAD_BLOCK_TABLE, or FA_ERR_INVALID_ARG for varlen offsets outside
 * the buffers) into *status.  Returns FA_ERR_CUDA if the
 * synchronisation itself failed.
 */
fa_status fa_get_device_status(void* stream, int* status);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
