// Cache write: scatter new tokens' rows into the paged latent pool.
//
// bf16 rows (1152 B) are concat(latent[0:512], k_pe[0:64]) ("sabi-mla-vllm"
// README, "What the plugin does"; vLLM PR #55543 commit 3.1+3.2,
// concat_and_cache_mla). fp8_ds_mla rows (656 B) hold the e4m3 codes of the
// latent divided by a per-128-block scale absmax/448, the four fp32 scales and
// the bf16 k_pe (vLLM PR #55543 commit 5.1-5.4 and PR description "Approach").
//
// One warp per token; every row offset is slot * row_bytes in 64-bit. A slot
// at or past num_slots is skipped on the device (nothing is written for that
// token) and, when the caller passes a status word, sets its bit 2: an
// out-of-range slot is the illegal memory access of the "sabi-mla-vllm"
// README, "B300 fix (0.2.0)", and the write must not reach past the pool.
#include "launch.cuh"
#include "mla_common.cuh"

namespace mla {

__global__ void __launch_bounds__(256) cache_write_bf16_kernel(const __nv_bfloat16* __restrict__ latent,
                                                               int64_t latent_stride,
                                                               const __nv_bfloat16* __restrict__ k_pe,
                                                               int64_t k_pe_stride,
                                                               const int64_t* __restrict__ slot_mapping,
                                                               int64_t num_tokens, uint8_t* __restrict__ cache,
                                                               int64_t num_slots, int* __restrict__ status) {
    const int64_t t = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= num_tokens) return;
    const int64_t slot = slot_mapping[t];
    if (slot < 0) return;
    if (slot >= num_slots) {
        if (lane == 0 && status) atomicOr(status, kErrBadBlock);
        return;
    }
    uint8_t* row = cache + slot * static_cast<int64_t>(kRowBf16);
    const uint4* src_l = reinterpret_cast<const uint4*>(latent + t * latent_stride);
    const uint4* src_r = reinterpret_cast<const uint4*>(k_pe + t * k_pe_stride);
    uint4* dst = reinterpret_cast<uint4*>(row);
    // 72 units of 16 bytes: 64 of latent, then 8 of k_pe
    const uint4 a = __ldg(src_l + lane);
    const uint4 b = __ldg(src_l + lane + 32);
    dst[lane] = a;
    dst[lane + 32] = b;
    if (lane < 8) dst[64 + lane] = __ldg(src_r + lane);
}

// bf16 rows of another latent width: concat(latent[0:D], k_pe[0:64]), D a
// multiple of 128 (2 (D + 64) bytes a row). One warp per token, 16-byte units.
__global__ void __launch_bounds__(256) cache_write_bf16_latent_kernel(const __nv_bfloat16* __restrict__ latent,
                                                                      int64_t latent_stride,
                                                                      const __nv_bfloat16* __restrict__ k_pe,
                                                                      int64_t k_pe_stride,
                                                                      const int64_t* __restrict__ slot_mapping,
                                                                      int64_t num_tokens, int D,
                                                                      uint8_t* __restrict__ cache, int64_t num_slots,
                                                                      int* __restrict__ status) {
    const int64_t t = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= num_tokens) return;
    const int64_t slot = slot_mapping[t];
    if (slot < 0) return;
    if (slot >= num_slots) {
        if (lane == 0 && status) atomicOr(status, kErrBadBlock);
        return;
    }
    const int lat_units = D / 8;  // 16-byte units of latent
    uint4* dst = reinterpret_cast<uint4*>(cache + slot * static_cast<int64_t>(2 * (D + kP)));
    const uint4* src_l = reinterpret_cast<const uint4*>(latent + t * latent_stride);
    const uint4* src_r = reinterpret_cast<const uint4*>(k_pe + t * k_pe_stride);
    for (int u = lane; u < lat_units; u += 32) dst[u] = __ldg(src_l + u);
    if (lane < kP / 8) dst[lat_units + lane] = __ldg(src_r + lane);
}

__global__ void __launch_bounds__(256) cache_write_fp8_kernel(const __nv_bfloat16* __restrict__ latent,
                                                              int64_t latent_stride,
                                                              const __nv_bfloat16* __restrict__ k_pe,
                                                              int64_t k_pe_stride,
                                                              const int64_t* __restrict__ slot_mapping,
                                                              int64_t num_tokens, uint8_t* __restrict__ cache,
                                                              int64_t num_slots, int* __restrict__ status) {
    const int64_t t = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= num_tokens) return;
    const int64_t slot = slot_mapping[t];
    if (slot < 0) return;
    if (slot >= num_slots) {
        if (lane == 0 && status) atomicOr(status, kErrBadBlock);
        return;
    }
    uint8_t* row = cache + slot * static_cast<int64_t>(kRowFp8);
    // lane owns latent values [16*lane, 16*lane+16); lanes 8j..8j+7 form block j
    const uint4* src = reinterpret_cast<const uint4*>(latent + t * latent_stride) + 2 * lane;
    uint4 raw[2] = {__ldg(src), __ldg(src + 1)};
    const __nv_bfloat16* xv = reinterpret_cast<const __nv_bfloat16*>(raw);
    float x[16];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        x[i] = __bfloat162float(xv[i]);
        amax = fmaxf(amax, fabsf(x[i]));
    }
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float scale = (amax == 0.f) ? 1.f : __fdiv_rn(amax, 448.f);
    uint32_t packed[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        uint32_t v = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float q = __fdiv_rn(x[4 * w + k], scale);
            const uint32_t code = __nv_cvt_float_to_fp8(q, __NV_SATFINITE, __NV_E4M3);
            v |= code << (8 * k);
        }
        packed[w] = v;
    }
    reinterpret_cast<uint4*>(row)[lane] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    if ((lane & 7) == 0) reinterpret_cast<float*>(row + 512)[lane >> 3] = scale;
    if (lane < 8) {
        const uint4 r = __ldg(reinterpret_cast<const uint4*>(k_pe + t * k_pe_stride) + lane);
        reinterpret_cast<uint4*>(row + 528)[lane] = r;
    }
}

// Prefill-context gather of an fp8_ds_mla pool into 576-wide bf16 rows (vLLM
// PR #55543: the fp8_ds_mla context-gather path, cp_gather_and_upconvert_fp8_
// kv_cache, fills a workspace whose rows must be 576 wide). Row r = cu[b] + j
// of dst gets request b's context token j: its 512 codes times their block
// scale (one fp32 multiply, then bf16 round to nearest even) and its 64 rope
// values as stored. One warp per row, kGatherRows consecutive rows per warp:
// their slots and loads go out before any row is converted.
constexpr int kGatherRows = 4;

__global__ void __launch_bounds__(256) gather_upconvert_fp8_kernel(const uint8_t* __restrict__ cache, int64_t num_slots,
                                                                   int page_size, const int32_t* __restrict__ block_table,
                                                                   int64_t bt_stride, const int32_t* __restrict__ cu,
                                                                   int B, int64_t num_rows,
                                                                   __nv_bfloat16* __restrict__ dst, int64_t dst_stride) {
    const int lane = threadIdx.x & 31;
    const int64_t r0 = (static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5)) * kGatherRows;
    if (r0 >= num_rows) return;
    // the request holding row r0: the last b with cu[b] <= r0 (cu is non-decreasing)
    int lo = 0, hi = B;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(cu + mid) <= r0) lo = mid;
        else hi = mid;
    }
    int b = lo;
    int64_t slot[kGatherRows];
    bool have[kGatherRows], ok[kGatherRows];
#pragma unroll
    for (int k = 0; k < kGatherRows; ++k) {
        const int64_t r = r0 + k;
        while (b < B && __ldg(cu + b + 1) <= r) ++b;
        const int64_t c0 = b < B ? __ldg(cu + b) : 0;
        have[k] = r < num_rows && b < B && r >= c0;
        ok[k] = false;
        slot[k] = 0;
        if (have[k]) {
            const int64_t j = r - c0;
            // a page index past the block-table row reads as an entry outside the pool
            const int64_t pi = j / page_size;
            const int64_t page = pi < bt_stride ? __ldg(block_table + static_cast<int64_t>(b) * bt_stride + pi) : -1;
            const int64_t s = page * page_size + j % page_size;
            ok[k] = page >= 0 && s < num_slots;
            slot[k] = ok[k] ? s : 0;
        }
    }
    uint4 codes[kGatherRows], rope[kGatherRows];
    float sc[kGatherRows];
#pragma unroll
    for (int k = 0; k < kGatherRows; ++k) {
        const uint8_t* row = cache + slot[k] * static_cast<int64_t>(kRowFp8);
        if (ok[k]) {
            codes[k] = __ldg(reinterpret_cast<const uint4*>(row) + lane);
            sc[k] = __ldg(reinterpret_cast<const float*>(row + 512) + (lane >> 3));
            if (lane < 8) rope[k] = __ldg(reinterpret_cast<const uint4*>(row + 528) + lane);
        }
    }
#pragma unroll
    for (int k = 0; k < kGatherRows; ++k) {
        if (!have[k]) continue;
        uint4* out = reinterpret_cast<uint4*>(dst + (r0 + k) * dst_stride);
        uint4 a = make_uint4(0u, 0u, 0u, 0u), c = a, e = a;
        if (ok[k]) {
            dequant16(codes[k], sc[k], a, c);
            if (lane < 8) e = rope[k];
        }
        out[2 * lane] = a;  // values 16 lane .. 16 lane + 15
        out[2 * lane + 1] = c;
        if (lane < 8) out[64 + lane] = e;
    }
}

cudaError_t launch_cache_write_latent(const void* latent, int64_t latent_stride, const void* k_pe,
                                      int64_t k_pe_stride, const int64_t* slot_mapping, int64_t num_tokens,
                                      void* cache, int64_t num_slots, int lat_dim, int* status,
                                      cudaStream_t stream) {
    if (num_tokens == 0) return cudaSuccess;
    const int64_t blocks = (num_tokens + 7) / 8;
    cache_write_bf16_latent_kernel<<<dim3(static_cast<unsigned>(blocks)), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(latent), latent_stride, static_cast<const __nv_bfloat16*>(k_pe), k_pe_stride,
        slot_mapping, num_tokens, lat_dim, static_cast<uint8_t*>(cache), num_slots, status);
    return cudaGetLastError();
}

cudaError_t launch_gather_upconvert(const void* cache, int64_t num_slots, int page_size, const int32_t* block_table,
                                    int64_t bt_stride, const int32_t* cu_seq_lens, int B, int64_t num_rows, void* dst,
                                    int64_t dst_stride, cudaStream_t stream) {
    if (num_rows == 0 || B == 0) return cudaSuccess;
    const int64_t blocks = (num_rows + 8 * kGatherRows - 1) / (8 * kGatherRows);
    gather_upconvert_fp8_kernel<<<dim3(static_cast<unsigned>(blocks)), 256, 0, stream>>>(
        static_cast<const uint8_t*>(cache), num_slots, page_size, block_table, bt_stride, cu_seq_lens, B, num_rows,
        static_cast<__nv_bfloat16*>(dst), dst_stride);
    return cudaGetLastError();
}

cudaError_t launch_cache_write(const void* latent, int64_t latent_stride, const void* k_pe, int64_t k_pe_stride,
                               const int64_t* slot_mapping, int64_t num_tokens, void* cache, int64_t num_slots,
                               int kind, int* status, cudaStream_t stream) {
    if (num_tokens == 0) return cudaSuccess;
    const int64_t blocks = (num_tokens + 7) / 8;
    const dim3 grid(static_cast<unsigned>(blocks));
    if (kind == 0)
        cache_write_bf16_kernel<<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(latent), latent_stride,
                                                          static_cast<const __nv_bfloat16*>(k_pe), k_pe_stride,
                                                          slot_mapping, num_tokens, static_cast<uint8_t*>(cache),
                                                          num_slots, status);
    else
        cache_write_fp8_kernel<<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(latent), latent_stride,
                                                         static_cast<const __nv_bfloat16*>(k_pe), k_pe_stride,
                                                         slot_mapping, num_tokens, static_cast<uint8_t*>(cache),
                                                         num_slots, status);
    return cudaGetLastError();
}

}  // namespace mla
