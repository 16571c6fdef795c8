/*
 * mla.h - C ABI of the GB300 (sm_103a) library for multi-head latent attention
 * (MLA) decode over a paged latent KV cache.
 *
 * Every pointer argument named "device" must point to memory the current CUDA
 * device can access (for example a torch CUDA tensor); "host" pointers are
 * ordinary CPU memory. The caller owns every buffer. Entry points validate
 * their arguments on the host, enqueue kernels on `stream` (a cudaStream_t;
 * NULL = the legacy default stream) and return without synchronising; they
 * never allocate memory. A non-zero return means nothing was enqueued, except
 * MLA_ERR_CUDA, which reports a failed launch.
 *
 * Cache geometry. Each cached token is one row of the paged pool:
 *   MLA_CACHE_BF16_576       1152 bytes: latent c[0:512] then k_pe[0:64], bf16.
 *                            ("sabi-mla-vllm" README: intro paragraph and "What
 *                            the plugin does": 512-d latent plus one shared
 *                            64-d rotary key, 576 values per token, paged bf16.)
 *   MLA_CACHE_FP8_DS_MLA_656 656 bytes: [0,512) e4m3 codes of c / scale_j,
 *                            [512,528) four fp32 scales scale_j = absmax_j/448
 *                            over the 128-value blocks j = d/128 (1.0 for an
 *                            all-zero block), [528,656) the 64 bf16 k_pe values.
 *                            (vLLM PR #55543, commits 3.1+3.2 and 5.1-5.4, PR
 *                            description "Approach" and "Memory tradeoff".)
 * The pool is addressed as [num_slots, row_bytes]; token j of request b lives
 * in slot block_table[b][j / page_size] * page_size + j % page_size. Every
 * offset is formed in 64-bit arithmetic, so slots above 2^31 / 576 =
 * 3,728,270 are read correctly ("sabi-mla-vllm" README, "B300 fix (0.2.0)").
 */
#ifndef MLA_GB300_H_
#define MLA_GB300_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MLA_API __attribute__((visibility("default")))
#else
#define MLA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MLA_OK = 0,
    MLA_ERR_INVALID_ARG = -1,  /* bad size, null or misaligned pointer */
    MLA_ERR_UNSUPPORTED = -2,  /* valid request this build does not handle */
    MLA_ERR_WORKSPACE = -3,    /* workspace too small */
    MLA_ERR_CUDA = -4,         /* a CUDA runtime call or launch failed */
    MLA_ERR_SCRATCH_LIMIT = -5 /* mla_decode_static_scratch: the call needs more
                                  than MLA_STATIC_SCRATCH_BYTES of scratch */
} mla_status;

enum { MLA_CACHE_BF16_576 = 0, MLA_CACHE_FP8_DS_MLA_656 = 1 };
enum { MLA_OUT_BF16 = 0, MLA_OUT_F32 = 1 };

/* Bytes of one cached row for a cache kind (1152 or 656), or 0 if unknown. */
MLA_API int mla_row_bytes(int cache_kind);

/*
 * mla_cache_write - scatter new tokens into the paged pool.
 * Follows vLLM PR #55543 commit 3.1+3.2 (concat_and_cache_mla: rows are
 * concat(latent, k_pe) with kv_lora_rank 512 and pe_dim 64; 656-byte rows for
 * fp8_ds_mla) and commit 5.1-5.4 (NoPE bytes are a per-128-block fp8
 * quantisation; rope bytes are the bf16 k_pe).
 *   latent        device, bf16 [num_tokens, 512], row stride latent_stride
 *                 elements (multiple of 8, base 16-byte aligned).
 *   k_pe          device, bf16 [num_tokens, 64], row stride k_pe_stride
 *                 elements (multiple of 8, base 16-byte aligned).
 *   slot_mapping  device, int64 [num_tokens]; a negative entry skips the token.
 *   cache         device, [num_slots, mla_row_bytes(cache_kind)] bytes, 16-byte
 *                 aligned. Rows not named by slot_mapping are left unchanged.
 *   num_slots     rows in the pool. A slot_mapping entry >= num_slots is
 *                 skipped on the device: nothing is written for that token,
 *                 so a bad slot cannot write past the pool (the out-of-range
 *                 access of "sabi-mla-vllm" README, "B300 fix (0.2.0)").
 *   status        device, one int32 (4-byte aligned), or NULL. When given,
 *                 the call ORs bit 2 (value 2, as in the decode status word)
 *                 into it if it skipped a slot >= num_slots; it never clears
 *                 it, so zero it before the calls it should cover.
 * fp8 rows: scale_j = absmax_j / 448 by IEEE fp32 division, each code is the
 * round-to-nearest-even, saturating e4m3 encoding of the fp32 quotient x /
 * scale_j. Two tokens mapped to the same slot race (the last write is
 * unspecified). Returns MLA_ERR_INVALID_ARG on bad sizes, pointers or strides.
 */
MLA_API int mla_cache_write(const void* latent, int64_t latent_stride, const void* k_pe, int64_t k_pe_stride,
                    const int64_t* slot_mapping, int64_t num_tokens, void* cache, int64_t num_slots,
                    int cache_kind, int32_t* status, void* stream);

/*
 * mla_gather_upconvert - the prefill-context gather of an fp8_ds_mla pool into
 * 576-wide bf16 rows (vLLM PR #55543, the commit that derives mla_dims from
 * the runtime layers and the PR description: the fp8_ds_mla context-gather
 * path, cp_gather_and_upconvert_fp8_kv_cache, fills a workspace whose rows
 * must be 576 wide). For request b < B and context token
 * j < cu_seq_lens[b+1] - cu_seq_lens[b]:
 *   slot = block_table[b][j / page_size] * page_size + j % page_size  (64-bit)
 *   dst[cu_seq_lens[b] + j][d]       = bf16(e4m3(code_d) * scale_{d/128}), d < 512
 *   dst[cu_seq_lens[b] + j][512 + e] = the row's rope value e as stored, e < 64
 * The product is one fp32 multiply (the e4m3 value widens exactly), rounded
 * to bf16 to nearest even.
 *   cache        device, the fp8_ds_mla pool written by mla_cache_write:
 *                num_slots rows of 656 bytes, 16-byte aligned.
 *   page_size    tokens per page, >= 1.
 *   block_table  device, int32 [B, block_table_stride]; entries past
 *                ceil(len_b / page_size) are never read, and a page index
 *                >= block_table_stride (a request longer than its row) counts
 *                as an entry outside the pool.
 *   cu_seq_lens  device, int32 [B + 1], non-decreasing, cu_seq_lens[0] = 0
 *                (read on the device only).
 *   num_rows     rows of dst the call may write (normally cu_seq_lens[B]);
 *                rows cu_seq_lens[b] + j >= num_rows are skipped.
 *   dst          device, bf16 [num_rows, dst_stride], 16-byte aligned,
 *                caller-owned; rows no request names are not touched.
 *   dst_stride   elements between rows, >= 576 and a multiple of 8.
 * A block-table entry outside the pool writes its row as zeros. Returns
 * MLA_ERR_INVALID_ARG for bad sizes or pointers (B = 0 or num_rows = 0 is a
 * no-op), MLA_ERR_CUDA if the launch fails. Does not synchronise.
 */
MLA_API int mla_gather_upconvert(const void* cache, int64_t num_slots, int page_size, const int32_t* block_table,
                                 int64_t block_table_stride, const int32_t* cu_seq_lens, int B, int64_t num_rows,
                                 void* dst, int64_t dst_stride, void* stream);

/*
 * mla_decode_workspace_bytes - bytes of device workspace mla_decode needs.
 *   B, q_len, Hq   as for mla_decode.
 *   num_ctas       the value that will be passed to mla_decode (0 = as many
 *                  CTAs as fit on the current device).
 * The workspace holds a 256-byte header (word 0: device-side status, see
 * mla_decode), one 64-byte status record per CTA, and fp32 partial results of
 * requests split across CTAs, each part rounded up to 256 bytes.
 * Returns 0 for invalid sizes.
 */
MLA_API size_t mla_decode_workspace_bytes(int B, int q_len, int Hq, int num_ctas);

/*
 * mla_decode - absorbed MLA decode over the paged latent cache.
 * For request b, query token t < q_len and head h, the row is
 * r = (b * q_len + t) * Hq + h and the visible tokens are j = 0 ..
 * seq_lens[b] - q_len + t (the q_len new tokens are already in the cache; each
 * sees itself and its past, as in the multi-token verify step of "qwen-mla-vllm"
 * README, "Speculative decoding (MTP)", which reads the latent once per
 * request). With c_j = row[0:512], k_pe_j = row[512:576] (fp8 rows:
 * c_j[d] = e4m3(code) * scale_{d/128}, widened in the kernel to f16 with the
 * latent queries and probabilities in f16 too up to 64 rows, to bf16 above):
 *   s_j      = scale * (q_lat[r] . c_j + q_pe[r] . k_pe_j)
 *   out[r]   = sum_j softmax_j(s) c_j          (softmax over the tokens)
 *   lse[r]   = ln sum_j exp(s_j)
 * A row with no visible token gets out = 0 and lse = -inf (vLLM PR #55543
 * commit 5.1-5.4: all-invalid rows neutralise to (0, -inf)).
 *   q_lat        device, bf16 [B*q_len, Hq, 512], contiguous, 16-byte aligned.
 *   q_pe         device, bf16 [B*q_len, Hq, 64], contiguous, 16-byte aligned.
 *   cache        device, the pool written by mla_cache_write, 16-byte aligned,
 *                num_slots rows of mla_row_bytes(cache_kind) bytes.
 *   page_size    tokens per page, >= 1.
 *   block_table  device, int32 [B, block_table_stride]; entries past
 *                ceil(seq_lens[b] / page_size) are never read. A request
 *                longer than its row (page index >= block_table_stride)
 *                reads nothing past the row: those page indices count as
 *                entries outside the pool.
 *   seq_lens     device, int32 [B], each >= 0; read on the device only, so the
 *                call does not synchronise.
 *   scale        softmax scale applied to the dot products.
 *   out          device, [B*q_len, Hq, 512], bf16 or fp32 per out_dtype.
 *   lse          device, fp32 [B*q_len, Hq], natural log.
 *   workspace    device, at least mla_decode_workspace_bytes(B, q_len, Hq,
 *                num_ctas) bytes, 256-byte aligned; needs no initialisation.
 *                Once the call's work has run, its first int32 holds
 *                device-side status bits: 1 = a bounded internal wait gave up
 *                (the kernel returned early, outputs are invalid), 2 = a
 *                block-table entry pointed outside the pool, or a page index
 *                was past the table row (page 0 was read instead), 4 = fp8 pools up to 64 rows, which compute in f16:
 *                a block scale above 146 or a query value above 65504 in
 *                magnitude was met (outputs may hold inf or NaN; the cache
 *                writer's scales stay below 146 for latents under 65,000 in
 *                magnitude). Words 1..3: wait site, tile and CTA of the lowest
 *                failing CTA; words 4..11 where each of its roles gave up.
 *                Calls sharing a workspace must be ordered on one stream.
 *   num_ctas     CTAs sharing the token stream (0 = as many as fit on the
 *                device, one per SM). Pools whose page_size is a multiple of
 *                8 (bf16 at any row count, fp8 up to 64 rows): each CTA is a
 *                worker on 64-token tiles of whole rows, except at 65..128
 *                rows (Hq * q_len), where the two 64-row groups of a worker
 *                are a cluster of two CTAs sharing each tile (num_ctas / 2
 *                workers). fp8 pools above 64 rows and page sizes that are
 *                not a multiple of 8: clusters of two CTAs that split each
 *                token's 576 dims between them, num_ctas / 2 workers on
 *                128-token tiles. The tiles of all requests are dealt out as
 *                equal contiguous ranges, one per worker; requests cut across
 *                workers are merged from fp32 partials by a second kernel.
 * Limits: Hq * q_len rows are processed in groups of at most 64; up to 128
 * rows (bf16 pools, page_size a multiple of 8) the cache is read once per
 * request, beyond that once per row group. Returns MLA_ERR_UNSUPPORTED on a
 * device other than sm_103 / sm_100 family.
 */
MLA_API int mla_decode(const void* q_lat, const void* q_pe, const void* cache, int cache_kind, int64_t num_slots,
               int page_size, const int32_t* block_table, int64_t block_table_stride, const int32_t* seq_lens,
               int B, int q_len, int Hq, float scale, void* out, int out_dtype, float* lse, void* workspace,
               size_t workspace_bytes, int num_ctas, void* stream);

/*
 * Other latent widths ("qwen-mla-vllm" README, "How it works": the
 * full-attention layers cache a per-layer latent of rank 256, 768 or 1792
 * plus a small rotary and normalisation tail). A row is bf16
 * [latent D | rope 64], 2 (D + 64) bytes; the normalisation is applied before
 * a row is cached, so the decode is mla_decode's definition with D latent
 * values in place of 512. D = 512 is the 576-wide row of mla_cache_write /
 * mla_decode.
 *
 * mla_cache_write_latent - mla_cache_write for bf16 rows of latent width
 * lat_dim (256, 512, 768 or 1792): latent [num_tokens, lat_dim] (row stride
 * latent_stride >= lat_dim, a multiple of 8), k_pe, slot_mapping, num_slots
 * and status as for mla_cache_write, cache [num_slots, 2 (lat_dim + 64)]
 * bytes, 16-byte aligned. Rows are bit copies.
 *
 * mla_decode_latent_workspace_bytes - the workspace of mla_decode_latent
 * (0 for invalid sizes): the mla_decode layout with lat_dim-wide partials.
 *
 * mla_decode_latent - mla_decode over such rows: q_lat [B*q_len, Hq, lat_dim],
 * q_pe [B*q_len, Hq, 64], out [B*q_len, Hq, lat_dim] (bf16 or fp32), lse
 * [B*q_len, Hq]; the visibility rule, the (0, -inf) rows, the status words
 * and every other argument as mla_decode with a bf16 pool. Each CTA works on
 * 64-token tiles whose rows are folded into two halves (as mla_decode's bf16
 * path at up to 32 query rows); at lat_dim 1792 the two CTAs of a cluster
 * each hold one 896-value half of every row and exchange partial scores.
 * Supported: lat_dim 512 wherever mla_decode takes a bf16 pool (it is that
 * call); lat_dim 256 with Hq * q_len <= 32 and lat_dim 768 or 1792 with
 * Hq * q_len <= 16, page_size a multiple of 8; otherwise MLA_ERR_UNSUPPORTED
 * before any launch.
 */
MLA_API int mla_cache_write_latent(const void* latent, int64_t latent_stride, const void* k_pe, int64_t k_pe_stride,
                                   const int64_t* slot_mapping, int64_t num_tokens, void* cache, int64_t num_slots,
                                   int lat_dim, int32_t* status, void* stream);
MLA_API size_t mla_decode_latent_workspace_bytes(int B, int q_len, int Hq, int lat_dim, int num_ctas);
MLA_API int mla_decode_latent(const void* q_lat, const void* q_pe, const void* cache, int lat_dim, int64_t num_slots,
                              int page_size, const int32_t* block_table, int64_t block_table_stride,
                              const int32_t* seq_lens, int B, int q_len, int Hq, float scale, void* out, int out_dtype,
                              float* lse, void* workspace, size_t workspace_bytes, int num_ctas, void* stream);

/*
 * mla_decode_varlen - mla_decode for a batch whose requests verify different
 * numbers of tokens (a chunked verify step: "qwen-mla-vllm" README,
 * "Speculative decoding (MTP)", a verify step of 1 + k tokens reads the latent
 * once per request; here k is per request). Request b verifies
 * q_len_b = cu_q_lens[b+1] - cu_q_lens[b] tokens, the last q_len_b of its
 * seq_lens[b]; its rows are r = (cu_q_lens[b] + t) * Hq + h (t < q_len_b) and
 * query t sees tokens 0 .. seq_lens[b] - q_len_b + t. Every other argument,
 * the outputs' layout (rows r above) and the status words are as mla_decode.
 *   total_q_tokens  cu_q_lens[B] (host copy): the query tokens in q_lat, q_pe,
 *                   out and lse.
 *   cu_q_lens       device, int32 [B + 1], non-decreasing, cu_q_lens[0] = 0,
 *                   every q_len_b <= max_q_len.
 *   max_q_len       the largest q_len_b, >= 1. Rows are processed in groups of
 *                   64 as in mla_decode with q_len = max_q_len; the workspace
 *                   is mla_decode_workspace_bytes(B, max_q_len, Hq, num_ctas).
 * While max_q_len * Hq <= 64, and up to 128 for bf16 pools whose page_size
 * is a multiple of 8 (two row groups sharing each tile), every request's
 * cache is read once. The kernels clamp every cu_q_lens entry to
 * [0, total_q_tokens], so no row at or past total_q_tokens * Hq of q_lat,
 * q_pe, out or lse is read or written whatever the prefix sums hold: a
 * request whose sums run past total_q_tokens verifies only its tokens below
 * it, with the length the clamped sums give (nothing flags this).
 */
MLA_API int mla_decode_varlen(const void* q_lat, const void* q_pe, int64_t total_q_tokens, const void* cache,
                              int cache_kind, int64_t num_slots, int page_size, const int32_t* block_table,
                              int64_t block_table_stride, const int32_t* seq_lens, const int32_t* cu_q_lens, int B,
                              int max_q_len, int Hq, float scale, void* out, int out_dtype, float* lse,
                              void* workspace, size_t workspace_bytes, int num_ctas, void* stream);

/*
 * mla_merge_lse - combine S partial results of the same N rows computed over
 * disjoint token sets (flash-decoding split-KV / decode context parallel
 * combine; vLLM PR #55543 commit 5.1-5.4 "(0, -inf) per the DCP merge
 * contract"):
 *   L      = ln sum_i exp(part_lse[i][n])
 *   out[n] = sum_i exp(part_lse[i][n] - L) * part_out[i][n]
 *   lse[n] = L;   rows whose partials are all -inf give (0, -inf).
 *   part_out  device, fp32 [S, N, 512], contiguous.
 *   part_lse  device, fp32 [S, N].
 *   out       device, [N, 512] bf16 or fp32 per out_dtype.
 *   lse       device, fp32 [N] (may be NULL).
 */
MLA_API int mla_merge_lse(const float* part_out, const float* part_lse, int S, int64_t N, void* out, int out_dtype,
                  float* lse, void* stream);

/* Number of SMs of the current device (what num_ctas = 0 means), or < 0. */
MLA_API int mla_num_sms(void);

/*
 * mla_decode_static_scratch - mla_decode with its workspace taken from a
 * scratch array that the library holds in device memory, for callers that
 * cannot allocate: a C host with no device allocator, or a serving loop that
 * must not call cudaMalloc on the decode path (cudaMalloc may synchronise the
 * device and stall the other streams). The source pages have no counterpart;
 * the operation is exactly mla_decode's, and every argument has the meaning
 * mla_decode gives it.
 *   MLA_STATIC_SCRATCH_BYTES bounds the scratch (one array per device, placed
 *   when the library's device code is loaded). A call whose
 *   mla_decode_workspace_bytes(B, q_len, Hq, num_ctas) exceeds it returns
 *   MLA_ERR_SCRATCH_LIMIT and launches nothing; pass a smaller num_ctas or
 *   use mla_decode with your own workspace.
 *   Nothing in the scratch has to start at zero: each CTA clears its own
 *   status record and the merge step rewrites the status header.
 *   The first call on a device looks the array up (cudaGetSymbolAddress, which
 *   may load the device code); make it before any stream capture. The address
 *   is kept per device ordinal for the life of the process, so the library
 *   must not be used across a cudaDeviceReset (or any other teardown of the
 *   device's primary context). Calls share one array per device, so calls
 *   that can overlap (different streams, or several host threads) race on
 *   it: order them on one stream.
 *   The device-side status words that mla_decode leaves in its workspace
 *   header land in the scratch here; mla_static_scratch_status copies them
 *   out.
 */
#define MLA_STATIC_SCRATCH_BYTES (64u << 20)
MLA_API int mla_decode_static_scratch(const void* q_lat, const void* q_pe, const void* cache, int cache_kind,
                                      int64_t num_slots, int page_size, const int32_t* block_table,
                                      int64_t block_table_stride, const int32_t* seq_lens, int B, int q_len, int Hq,
                                      float scale, void* out, int out_dtype, float* lse, int num_ctas, void* stream);

/*
 * mla_static_scratch_status - copy the first n (1..12) int32 status words of
 * the static scratch into dst, in stream order: after the last
 * mla_decode_static_scratch call on this device they are the words
 * mla_decode documents for its workspace header (word 0: bit 1 = a bounded
 * wait gave up and the outputs are invalid, bit 2 = a block-table entry
 * outside the pool, bit 4 = an fp8 value past the f16 range; words 1..11
 * where). dst is device memory or pinned host
 * memory (one cudaMemcpyAsync, direction inferred); it allocates nothing.
 * Before any static-scratch call on the device the words are undefined.
 * Returns MLA_ERR_INVALID_ARG for a null dst or n outside 1..12.
 */
MLA_API int mla_static_scratch_status(int32_t* dst, int n, void* stream);

/*
 * mla_test_hold_next_decode - test support for the device-side failure path.
 * The next mla_decode call in this process withholds its first hand-off from
 * the softmax warps to the PV issuers, so their bounded wait gives up after
 * about one second: the call's status word then has bit 1 set (words 1..11
 * name the wait site and role), its outputs are invalid, and the device
 * context stays usable. Nothing else sets it; it has no other effect.
 */
MLA_API void mla_test_hold_next_decode(void);

/*
 * mla_test_slow_pv_next_decode - test support for the softmax -> PV hand-off.
 * In the next mla_decode call in this process, one of the two warps that
 * issue the value products (PV) busy-waits about 20 microseconds after each
 * of its first 32 tiles, so the softmax warps run up to two tiles ahead of it.
 * The call's results and status are those of an undelayed call; only its
 * duration grows. Nothing else sets it.
 */
MLA_API void mla_test_slow_pv_next_decode(void);

/* Static English text for a status code. */
MLA_API const char* mla_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* MLA_GB300_H_ */
