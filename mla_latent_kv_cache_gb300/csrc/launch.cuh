// Internal launch interface shared by the C ABI layer and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mla {

// Per-CTA status record (int32 words): 0 status bits, 1 first wait site,
// 2 its tile, 4 + role: (site << 24) | tile where that role gave up.
constexpr int kStatusRecWords = 16;

// Everything a decode launch needs; passed by value as a kernel parameter.
struct DecodeParams {
    const __nv_bfloat16* q_lat;
    const __nv_bfloat16* q_pe;
    const uint8_t* cache;
    int64_t num_slots;
    const int32_t* block_table;
    int64_t bt_stride;
    const int32_t* seq_lens;
    void* out;
    float* lse;
    int* status;       // workspace header: status summary written by the merge step
    int* rec;          // [CTAs][kStatusRecWords] per-CTA status records
    float* part_o;     // [GY][SPG][64][lat_dim] fp32 partial outputs
    float* part_lse;   // [GY][SPG][64] fp32 partial LSEs
    float scale_log2;  // softmax scale * log2(e)
    int page_size;
    int run_rows;      // TMA box height: gcd(page_size, tile)
    int tile_shift;    // log2 of the tokens per tile: 7 (cluster kernel) or 6 (folded tiles)
    int B, Qt, Hq, HQ; // HQ = Hq * Qt rows per request (the largest Qt when cu_q is given)
    int out_f32;
    int SPG;           // partial slots per row group = workers + B
    int wseg;          // work-split cost of a request boundary, in tiles
    int test_hold;     // test hooks: 1 = withhold the first hand-off to the PV issuers,
                       // 2 = hold one PV issuer ~20 us after each of its first 32 tiles
    const int32_t* cu_q;  // [B + 1] prefix sums of query tokens per request, or null: Qt each
    int total_q;          // query tokens in q_lat, q_pe, out and lse; cu_q is clamped to [0, total_q]
    int lat_dim;       // latent width D: 512 (576-value rows), or 256 / 768 / 1792 (folded tiles, bf16)
    int rope_dim;      // rotary width P: 64
};

cudaError_t launch_cache_write(const void* latent, int64_t latent_stride, const void* k_pe, int64_t k_pe_stride,
                               const int64_t* slot_mapping, int64_t num_tokens, void* cache, int64_t num_slots,
                               int kind, int* status, cudaStream_t stream);
// bf16 rows of another latent width D (2 (D + 64) bytes) (mla_cache_write_latent).
cudaError_t launch_cache_write_latent(const void* latent, int64_t latent_stride, const void* k_pe,
                                      int64_t k_pe_stride, const int64_t* slot_mapping, int64_t num_tokens,
                                      void* cache, int64_t num_slots, int lat_dim, int* status, cudaStream_t stream);
// Context gather of an fp8_ds_mla pool into bf16 rows (mla_gather_upconvert).
cudaError_t launch_gather_upconvert(const void* cache, int64_t num_slots, int page_size, const int32_t* block_table,
                                    int64_t bt_stride, const int32_t* cu_seq_lens, int B, int64_t num_rows, void* dst,
                                    int64_t dst_stride, cudaStream_t stream);
// Clusters (of 2 CTAs) the decode kernel variant runs with: the number that
// fit on the current device at once, or requested_ctas / 2 when given.
int decode_clusters(int NP, bool lsu, int kind, int requested_ctas);
// TMA descriptors of one decode call, unused when the load/convert warps
// read the pool. bf16 pools: lat = 64-dim latent chunks (128-B swizzle),
// rope = 32-dim rope halves (64-B swizzle). fp8 pools: lat = 256 code bytes
// of a row, aux = its 16 scale bytes, rope = 32-dim rope halves. q / qpe:
// 64-dim chunks of q_lat and 32-dim halves of q_pe, NP rows high.
struct DecodeMaps {
    CUtensorMap lat, aux, rope, q, qpe;
};

// Whether the folded-tile kernel has a variant for NP query rows, this latent
// width, cache kind and number of row groups.
bool fold_supported(int NP, int lat_dim, int kind, int GY);
// Whether that variant's workers are clusters of two CTAs (latent 1792).
bool fold_is_pair(int lat_dim);
// Workers of the folded-tile decode kernel (bf16 pools, page_size % 8 == 0)
// for GY row groups: the number that fit at once, or what requested_ctas CTAs
// make (a worker is a cluster of two for latent 1792, and for 65..128 query
// rows of the 576-wide row, whose two row groups share each tile).
int decode_fold_ctas(int NP, int lat_dim, int kind, int GY, int requested_ctas);
cudaError_t launch_decode_fold(const DecodeMaps& maps, const DecodeParams& p, int NP, int kind, int W, int GY,
                               cudaStream_t stream);
cudaError_t launch_decode(const DecodeMaps& maps, const DecodeParams& p, int NP, bool lsu, int kind, int G, int GY,
                          cudaStream_t stream);
cudaError_t launch_merge_lse(const float* part_o, const float* part_lse, int S, int64_t N, void* out, int out_f32,
                             float* lse, cudaStream_t stream);

}  // namespace mla
